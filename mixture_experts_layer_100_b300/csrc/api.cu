// C ABI of the MoE layer library: argument checks and the launch sequence
// of each entry point (see moe.h); the stages themselves are in stages.cu.
#include <cstring>
#include <mutex>
#include <vector>

#include "kernels.cuh"
#include "moe.h"
#include "stages.cuh"

using namespace moe;
using namespace moe::stage;

namespace {

moe_status check_config(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d <= 0 || c->E <= 0 || c->G <= 0 || c->K <= 0 || c->M <= 0 || c->I <= 0 || c->S < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->E % c->G != 0 || c->G > 32 || c->M > c->G) return MOE_ERR_INVALID_ARG;
  const int gsz = c->E / c->G;
  if (c->group_topk < 1 || c->group_topk > gsz) return MOE_ERR_INVALID_ARG;
  if (c->K > 32 || c->K > c->M * gsz) return MOE_ERR_INVALID_ARG;
  if (c->E > 512) return MOE_ERR_UNSUPPORTED;
  if (c->act != MOE_F32 && c->act != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->expert != c->act && !(is_f8(c->expert) && c->act == MOE_BF16)) return MOE_ERR_INVALID_ARG;
  if ((long long)c->T * c->K > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  if (c->combine != MOE_COMBINE_GATHER && c->combine != MOE_COMBINE_SCATTER_ADD) return MOE_ERR_INVALID_ARG;
  if (c->act == MOE_BF16) {
    if (c->d % 128 != 0 || c->I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (c->E > 256) return MOE_ERR_UNSUPPORTED;
    if (is_f8(c->expert) && c->d % 256 != 0) return MOE_ERR_UNSUPPORTED;
  } else if (c->d % 128 != 0 || c->I % 128 != 0) {
    return MOE_ERR_UNSUPPORTED;  // fp32 layers run the same tcgen05 tiles (as tf32 pairs)
  }
  return MOE_OK;
}

moe_status check_weights(const moe_config& c, const moe_weights* w, bool routed, bool shared) {
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  if (routed && (!w->w13 || !w->w2 || !aligned16(w->w13) || !aligned16(w->w2))) return MOE_ERR_INVALID_ARG;
  if (shared && c.S > 0 && (!w->ws13 || !w->ws2 || !aligned16(w->ws13) || !aligned16(w->ws2)))
    return MOE_ERR_INVALID_ARG;
  if (is_f8(c.expert)) {
    if (routed && (!w->w13_scale || !w->w2_scale)) return MOE_ERR_INVALID_ARG;
    if (shared && c.S > 0 && (!w->ws13_scale || !w->ws2_scale)) return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

moe_status quantize_weights(const void* w, int n_mat, int rows, int cols, uint8_t* q, float* scale, bool ue8m0,
                            cudaStream_t st) {
  if (n_mat < 0 || rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
  if (n_mat == 0 || rows == 0 || cols == 0) return MOE_OK;
  if (!ok_ptr(w) || !ok_ptr(q) || scale == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(launch_quantize_blocks(static_cast<const __nv_bfloat16*>(w), n_mat, rows, cols, q, scale, ue8m0, st));
  return MOE_OK;
}

// Side stream of moe_layer_forward (one per host thread and device, created
// on first use and kept for the life of the process): the shared experts'
// GEMM1 runs there while the main stream routes and permutes.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

moe_status side_stream(SideStream** out) {
  thread_local SideStream cache[64];
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  SideStream& ss = cache[dev];
  if (ss.s == nullptr) {
    MOE_CUDA(cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking));
    MOE_CUDA(cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming));
    MOE_CUDA(cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming));
  }
  *out = &ss;
  return MOE_OK;
}

thread_local cudaEvent_t g_stage_events[8];
thread_local bool g_stage_on = false;
thread_local bool g_capturing = false;  // moe_layer_forward is being captured into a graph

moe_status stage_mark(int i, cudaStream_t st) {
  if (!g_stage_on) return MOE_OK;
  // inside a capture the record becomes a graph node (re-targeted at replay)
  if (g_capturing) {
    MOE_CUDA(cudaEventRecordWithFlags(g_stage_events[i], st, cudaEventRecordExternal));
  } else {
    MOE_CUDA(cudaEventRecord(g_stage_events[i], st));
  }
  return MOE_OK;
}

moe_status layer_forward_body(const moe_config& c, const void* x, const moe_weights* w, float* bias, float gamma,
                              void* out, int32_t* topk_idx, float* topk_gate, int32_t* counts, float* max_over_mean,
                              void* ws, cudaStream_t st);

// ---- CUDA-graph replay of moe_layer_forward. A call with the same
// configuration, buffers, gamma and stage-event setting as an earlier one on
// the same context replays the kernels captured at the second such call
// (same kernels, same arguments, so the same bits) instead of launching them
// one by one. Up to kMaxGraphs argument sets are kept; a new one replaces the
// least recently used (its executable graph is freed once any replay in
// flight has finished).
constexpr int kMaxGraphs = 16;

struct LayerKey {
  void* ctx;
  moe_config cfg;
  moe_weights w;
  const void* x;
  float* bias;
  uint32_t gamma_bits;
  void* out;
  int32_t* idx;
  float* gate;
  int32_t* counts;
  float* mom;
  void* ws;
  int stage_on;
};

struct LayerGraph {
  LayerKey key;
  unsigned long long last_use = 0;
  int calls = 0;
  bool failed = false;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t stage_nodes[8] = {};
};

std::mutex g_graph_mu;
std::vector<LayerGraph>* g_graphs = new std::vector<LayerGraph>();  // never freed: outlives static teardown
unsigned long long g_graph_clock = 0;

void release_graph(LayerGraph& g) {
  if (g.exec != nullptr) cudaGraphExecDestroy(g.exec);  // deferred by CUDA while a launch is in flight
  if (g.graph != nullptr) cudaGraphDestroy(g.graph);
  g = LayerGraph();
}
int g_graphs_mode = -1;  // -1: from MOE_LAYER_GRAPHS (default on), 0 off, 1 on

bool layer_graphs_on() {
  if (g_graphs_mode < 0) {
    const char* v = getenv("MOE_LAYER_GRAPHS");
    g_graphs_mode = (v != nullptr && v[0] == '0') ? 0 : 1;
  }
  return g_graphs_mode == 1;
}

void* current_context() {
  using Fn = int (*)(void**);
  static Fn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(p);
  }
  void* ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// Stream the captures are recorded on (one per host thread and device).
moe_status capture_stream(cudaStream_t* out) {
  thread_local cudaStream_t cache[64] = {};
  int dev = 0;
  MOE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  if (cache[dev] == nullptr) MOE_CUDA(cudaStreamCreateWithFlags(&cache[dev], cudaStreamNonBlocking));
  *out = cache[dev];
  return MOE_OK;
}

moe_status capture_layer(LayerGraph& g, const moe_config& c, const void* x, const moe_weights* w, float* bias,
                         float gamma, void* out, int32_t* idx, float* gate, int32_t* counts, float* mom, void* ws) {
  cudaStream_t cap = nullptr;
  MOE_TRY(capture_stream(&cap));
  MOE_CUDA(cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal));
  g_capturing = true;
  const moe_status s = layer_forward_body(c, x, w, bias, gamma, out, idx, gate, counts, mom, ws, cap);
  g_capturing = false;
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(cap, &graph);
  if (s != MOE_OK || e != cudaSuccess || graph == nullptr) {
    if (graph != nullptr) cudaGraphDestroy(graph);
    (void)cudaGetLastError();
    return s != MOE_OK ? s : MOE_ERR_CUDA;
  }
  if (cudaGraphInstantiate(&g.exec, graph, 0) != cudaSuccess) {
    g.exec = nullptr;
    cudaGraphDestroy(graph);
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  g.graph = graph;
  if (g.key.stage_on) {
    // the stage-event record nodes, to point them at each call's events
    size_t n = 0;
    MOE_CUDA(cudaGraphGetNodes(graph, nullptr, &n));
    std::vector<cudaGraphNode_t> nodes(n);
    MOE_CUDA(cudaGraphGetNodes(graph, nodes.data(), &n));
    for (cudaGraphNode_t node : nodes) {
      cudaGraphNodeType t;
      MOE_CUDA(cudaGraphNodeGetType(node, &t));
      if (t != cudaGraphNodeTypeEventRecord) continue;
      cudaEvent_t ev = nullptr;
      MOE_CUDA(cudaGraphEventRecordNodeGetEvent(node, &ev));
      for (int i = 0; i < 8; ++i)
        if (ev == g_stage_events[i] && g.stage_nodes[i] == nullptr) {
          g.stage_nodes[i] = node;
          break;
        }
    }
  }
  return MOE_OK;
}

moe_status replay_layer(LayerGraph& g, cudaStream_t st) {
  if (g.key.stage_on) {
    for (int i = 0; i < 8; ++i)
      if (g.stage_nodes[i] != nullptr)
        MOE_CUDA(cudaGraphExecEventRecordNodeSetEvent(g.exec, g.stage_nodes[i], g_stage_events[i]));
  }
  MOE_CUDA(cudaGraphLaunch(g.exec, st));
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  MOE_TRY(check_config(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = layout(*cfg).total;
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const void* x, const void* w_router, const float* scores_in,
                     const float* bias, float* scores_out, int32_t* topk_idx, float* topk_gate, int32_t* counts,
                     void* ws, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (!ok_ptr(bias) || !ok_ptr(topk_idx) || !ok_ptr(topk_gate) || !ok_ptr(counts) || !ok_ptr(ws))
    return MOE_ERR_INVALID_ARG;
  if (scores_in != nullptr && !aligned16(scores_in)) return MOE_ERR_INVALID_ARG;
  if (scores_out != nullptr && !aligned16(scores_out)) return MOE_ERR_INVALID_ARG;
  if (scores_in == nullptr && c.T > 0 && (!ok_ptr(x) || !ok_ptr(w_router))) return MOE_ERR_INVALID_ARG;
  return route_stage(c, x, w_router, scores_in, bias, scores_out, topk_idx, topk_gate, counts, ws,
                     reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_permute(const moe_config* cfg, const int32_t* topk_idx, const int32_t* counts, int32_t* offsets,
                       int32_t* sorted_tok, int32_t* slot_pos, const void* x, void* xp, float* xp_scale, void* ws,
                       moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (!ok_ptr(offsets) || !ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && (!ok_ptr(topk_idx) || !ok_ptr(counts) || !ok_ptr(sorted_tok) || !ok_ptr(slot_pos) || !ok_ptr(x) ||
                  !ok_ptr(xp)))
    return MOE_ERR_INVALID_ARG;
  if (is_f8(c.expert) && c.T > 0 && !ok_ptr(xp_scale)) return MOE_ERR_INVALID_ARG;
  return permute_stage(c, topk_idx, counts, offsets, sorted_tok, slot_pos, x, xp, xp_scale, nullptr, nullptr, ws,
                       reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_grouped_ffn(const moe_config* cfg, const void* xp, const float* xp_scale, const int32_t* offsets,
                           const moe_weights* w, void* yp, void* ws, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_weights(c, w, true, false));
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if (!ok_ptr(xp) || !ok_ptr(offsets) || !ok_ptr(yp)) return MOE_ERR_INVALID_ARG;
  if (is_f8(c.expert) && !ok_ptr(xp_scale)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (c.act == MOE_F32) {
    // the caller's fp32 rows and the expert weights as tf32 pairs
    void* xps = at<void>(ws, layout(c).xp);
    MOE_TRY(split_rows_f32(xp, (long long)c.T * c.K, c.d, xps, st));
    MOE_TRY(split_weights_f32(c, w, false, true, false, ws, st));
    xp = xps;
  }
  MOE_TRY(gemm1_stage(c, xp, xp_scale, offsets, nullptr, w, true, false, ws, st));
  MOE_TRY(gemm2_routed_stage(c, offsets, w, yp, ws, st));
  return MOE_OK;
}

moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* slot_pos, const float* topk_gate,
                       const void* x, const moe_weights* w, void* out, void* ws, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_weights(c, w, false, true));
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if (!ok_ptr(yp) || !ok_ptr(slot_pos) || !ok_ptr(topk_gate) || !ok_ptr(out)) return MOE_ERR_INVALID_ARG;
  if (c.S > 0 && !ok_ptr(x)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (c.S > 0) {
    if (c.act == MOE_F32) {
      void* xs = at<void>(ws, layout(c).xs);
      MOE_TRY(split_rows_f32(x, c.T, c.d, xs, st));
      MOE_TRY(split_weights_f32(c, w, false, false, true, ws, st));
      x = xs;
    }
    if (is_f8(c.expert)) {
      const Layout Lw = layout(c);
      MOE_CUDA(launch_quantize_rows(static_cast<const __nv_bfloat16*>(x), c.T, c.d, at<uint8_t>(ws, Lw.xq),
                                    at<float>(ws, Lw.xq_scale), c.expert == MOE_E4M3_UE8M0, num_sms(), st));
    }
    MOE_TRY(gemm1_stage(c, nullptr, nullptr, nullptr, x, w, false, true, ws, st));
  }
  MOE_TRY(gemm2_combine_stage(c, yp, slot_pos, topk_gate, w, out, ws, st));
  return MOE_OK;
}

moe_status moe_bias_update(const moe_config* cfg, const int32_t* counts, float gamma, float* bias,
                           float* max_over_mean, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (!ok_ptr(counts) || !ok_ptr(bias)) return MOE_ERR_INVALID_ARG;
  if (max_over_mean != nullptr && (reinterpret_cast<uintptr_t>(max_over_mean) & 3u)) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  MOE_CUDA(launch_bias_update(counts, c.E, (long long)c.T * c.K, gamma, bias, max_over_mean,
                              reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_layer_forward(const moe_config* cfg, const void* x, const moe_weights* w, float* bias, float gamma,
                             void* out, int32_t* topk_idx, float* topk_gate, int32_t* counts, float* max_over_mean,
                             void* ws, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  MOE_TRY(check_weights(c, w, true, true));
  if (!ok_ptr(bias) || !ok_ptr(counts) || !ok_ptr(ws) || !ok_ptr(topk_idx) || !ok_ptr(topk_gate))
    return MOE_ERR_INVALID_ARG;
  if (c.T > 0 && (!ok_ptr(x) || !ok_ptr(out) || !ok_ptr(w->w_router))) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (c.T > 0 && layer_graphs_on()) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    MOE_CUDA(cudaStreamIsCapturing(st, &cs));
    if (cs == cudaStreamCaptureStatusNone) {  // (a caller's own capture records the kernels themselves)
      LayerKey k;
      memset(&k, 0, sizeof(k));
      k.ctx = current_context();
      k.cfg = c;
      k.w = *w;
      k.x = x;
      k.bias = bias;
      memcpy(&k.gamma_bits, &gamma, sizeof(float));
      k.out = out;
      k.idx = topk_idx;
      k.gate = topk_gate;
      k.counts = counts;
      k.mom = max_over_mean;
      k.ws = ws;
      k.stage_on = g_stage_on ? 1 : 0;
      std::lock_guard<std::mutex> lock(g_graph_mu);
      LayerGraph* g = nullptr;
      for (LayerGraph& e : *g_graphs)
        if (memcmp(&e.key, &k, sizeof(k)) == 0) g = &e;
      if (g == nullptr && k.ctx != nullptr) {
        if ((int)g_graphs->size() < kMaxGraphs) {
          g_graphs->reserve(kMaxGraphs);  // entries never move
          g_graphs->emplace_back();
          g = &g_graphs->back();
        } else {
          g = &(*g_graphs)[0];
          for (LayerGraph& e : *g_graphs)
            if (e.last_use < g->last_use) g = &e;
          release_graph(*g);
        }
        g->key = k;
      }
      if (g != nullptr) g->last_use = ++g_graph_clock;
      if (g != nullptr && !g->failed) {
        if (g->exec == nullptr && ++g->calls >= 2) {
          // first repeat of this argument set: capture it (the first call ran
          // eagerly and set up the side stream, smem limits and tensor-map
          // encoder outside any capture)
          if (capture_layer(*g, c, x, w, bias, gamma, out, topk_idx, topk_gate, counts, max_over_mean, ws) !=
              MOE_OK)
            g->failed = true;
        }
        if (g->exec != nullptr) {
          const moe_status r = replay_layer(*g, st);
          if (r == MOE_OK) return MOE_OK;
          g->failed = true;  // run this call eagerly below
          (void)cudaGetLastError();
        }
      }
    }
  }
  return layer_forward_body(c, x, w, bias, gamma, out, topk_idx, topk_gate, counts, max_over_mean, ws, st);
}

moe_status moe_set_layer_graphs(int enable) {
  if (enable != 0 && enable != 1) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_graph_mu);
  g_graphs_mode = enable;
  return MOE_OK;
}

moe_status moe_layer_graphs_kept(int* n) {
  if (n == nullptr) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_graph_mu);
  int c = 0;
  for (const LayerGraph& e : *g_graphs) c += e.exec != nullptr;
  *n = c;
  return MOE_OK;
}

}  // extern "C"

namespace {

moe_status layer_forward_body(const moe_config& c, const void* x, const moe_weights* w, float* bias, float gamma,
                              void* out, int32_t* topk_idx, float* topk_gate, int32_t* counts, float* max_over_mean,
                              void* ws, cudaStream_t st) {
  const Layout Lw = layout(c);
  MOE_TRY(stage_mark(0, st));
  MOE_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, st));
  if (c.T > 0) {
    float* scores = at<float>(ws, Lw.scores);
    const bool f8 = is_f8(c.expert);
    const bool f32 = c.act == MOE_F32;
    const void* w_router = w->w_router;
    if (f32) {
      // fp32 layer: x and every weight as tf32 pairs for the tensor cores
      void* xs = at<void>(ws, Lw.xs);
      MOE_TRY(split_rows_f32(x, c.T, c.d, xs, st));
      MOE_TRY(split_weights_f32(c, w, true, true, true, ws, st));
      x = xs;
      w_router = f32_weights(c, ws).wr;
    }
    MOE_TRY(router_scores(c, x, w_router, scores, ws, st));
    MOE_TRY(stage_mark(1, st));
    // The shared experts' GEMM1 depends on x only: it runs on a side stream,
    // overlapping the memory-bound selection and permutation below; the main
    // stream waits for it before the shared down projection. With the
    // scatter-add combine the side stream also runs the shared down
    // projection, which writes the fp32 accumulator (zeros when S = 0), and
    // the main stream waits before the routed down projection adds into it.
    const bool scat = scatter_combine(c);
    float* acc = f32 ? static_cast<float*>(out) : at<float>(ws, Lw.acc);  // fp32 layers add into out itself
    SideStream* side = nullptr;
    if (c.S > 0 || scat) {
      MOE_TRY(side_stream(&side));
      MOE_CUDA(cudaEventRecord(side->fork, st));
      MOE_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
      if (f8 && c.S > 0) {
        MOE_CUDA(launch_quantize_rows(static_cast<const __nv_bfloat16*>(x), c.T, c.d, at<uint8_t>(ws, Lw.xq),
                                      at<float>(ws, Lw.xq_scale), c.expert == MOE_E4M3_UE8M0, num_sms(),
                                      side->s));
      }
      if (c.S > 0) MOE_TRY(gemm1_stage(c, nullptr, nullptr, nullptr, x, w, false, true, ws, side->s));
      if (scat) MOE_TRY(shared_seed_stage(c, w, acc, ws, side->s));
      MOE_CUDA(cudaEventRecord(side->join, side->s));
    }
    MOE_CUDA(launch_route_select(scores, bias, c.T, c.E, c.G, c.K, c.M, c.group_topk, topk_idx, topk_gate, counts,
                                 num_sms(), st));
    MOE_TRY(stage_mark(2, st));
    int32_t* offsets = at<int32_t>(ws, Lw.offsets);
    int32_t* slot_pos = at<int32_t>(ws, Lw.slot_pos);
    void* xp = at<void>(ws, Lw.xp);
    void* yp = at<void>(ws, Lw.yp);
    // padded layout (zero_padded): experts start at multiples of 128, zero rows between
    const bool padded = zero_padded(c);
    const int rows = expert_rows(c);
    MOE_TRY(permute_stage(c, topk_idx, counts, offsets, at<int32_t>(ws, Lw.sorted_tok), slot_pos, x, xp,
                          f8 ? at<float>(ws, Lw.xp_scale) : nullptr, nullptr, nullptr, ws, st,
                          scat ? topk_gate : nullptr, scat ? at<float>(ws, Lw.gate_p) : nullptr, f32,
                          padded ? 128 : 1));
    MOE_TRY(stage_mark(3, st));
    MOE_TRY(gemm1_stage(c, xp, f8 ? at<float>(ws, Lw.xp_scale) : nullptr, offsets, x, w, true, false, ws, st,
                        rows));
    MOE_TRY(stage_mark(4, st));
    if (scat) {
      MOE_CUDA(cudaStreamWaitEvent(st, side->join, 0));
      MOE_TRY(gemm2_scatter_stage(c, offsets, w, acc, ws, st));
      MOE_TRY(stage_mark(5, st));
      if (!f32) MOE_TRY(acc_round_stage(c, acc, out, st));
    } else {
      MOE_TRY(gemm2_routed_stage(c, offsets, w, yp, ws, st, rows, padded ? counts : nullptr));
      MOE_TRY(stage_mark(5, st));
      if (side != nullptr) MOE_CUDA(cudaStreamWaitEvent(st, side->join, 0));
      MOE_TRY(gemm2_combine_stage(c, yp, slot_pos, topk_gate, w, out, ws, st));
    }
    MOE_TRY(stage_mark(6, st));
    if (gamma != 0.0f)
      MOE_CUDA(launch_bias_update(counts, c.E, (long long)c.T * c.K, gamma, bias, max_over_mean, st));
    MOE_TRY(stage_mark(7, st));
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_quantize_weights_e4m3(const void* w, int n_mat, int rows, int cols, uint8_t* q, float* scale,
                                     moe_stream_t stream) {
  return quantize_weights(w, n_mat, rows, cols, q, scale, false, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_quantize_weights_e4m3_ue8m0(const void* w, int n_mat, int rows, int cols, uint8_t* q, float* scale,
                                           moe_stream_t stream) {
  return quantize_weights(w, n_mat, rows, cols, q, scale, true, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_seq_balance(const moe_config* cfg, const float* scores, const int32_t* topk_idx, int seq_len,
                           float alpha, float* loss, float* f, float* p, void* ws, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  const moe_config& c = *cfg;
  if (seq_len <= 0) return MOE_ERR_INVALID_ARG;
  if (c.T == 0) return MOE_OK;
  if (scores == nullptr) {
    if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
    scores = at<float>(ws, layout(c).scores);
  }
  if (!aligned16(scores) || !ok_ptr(topk_idx) || loss == nullptr) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(loss) | reinterpret_cast<uintptr_t>(f) | reinterpret_cast<uintptr_t>(p)) & 3u)
    return MOE_ERR_INVALID_ARG;
  MOE_CUDA(launch_seq_balance(scores, topk_idx, c.T, c.E, c.K, seq_len, alpha, loss, f, p,
                              reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

static moe_status move_rows(const void* src, const int32_t* idx, int n, int n_other, size_t row_bytes, void* dst,
                            bool gather, void* ws, moe_stream_t stream) {
  if (n < 0 || n_other < 0 || row_bytes == 0 || row_bytes % 4 != 0 || row_bytes / 4 > 0x7fffffffu ||
      ws == nullptr || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!ok_ptr(src) || !ok_ptr(dst) || !ok_ptr(idx)) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(launch_move_rows(src, idx, n, n_other, row_bytes, dst, gather, static_cast<int*>(ws), num_sms(),
                            reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_gather_rows(const void* src, int n_src, const int32_t* idx, int n, size_t row_bytes, void* dst,
                           void* ws, moe_stream_t stream) {
  return move_rows(src, idx, n, n_src, row_bytes, dst, true, ws, stream);
}

moe_status moe_scatter_rows(const void* src, const int32_t* idx, int n, size_t row_bytes, void* dst, int n_dst,
                            void* ws, moe_stream_t stream) {
  return move_rows(src, idx, n, n_dst, row_bytes, dst, false, ws, stream);
}

moe_status moe_set_stage_events(void* const* events, int count) {
  if (count == 0) {
    g_stage_on = false;
    return MOE_OK;
  }
  if (events == nullptr || count < 8) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 8; ++i)
    if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;  // the previous hook stays as it was
  for (int i = 0; i < 8; ++i) g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
  g_stage_on = true;
  return MOE_OK;
}

moe_status moe_device_error(void* ws, moe_stream_t stream, int* code) {
  if (ws == nullptr || code == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaStreamSynchronize(st));
  int v = 0;
  MOE_CUDA(cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost));
  *code = v;
  if (v != 0) {
    MOE_CUDA(cudaMemset(ws, 0, sizeof(int)));
    return (v & 0xF00) == 0x100 ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE;
  }
  return MOE_OK;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

}  // extern "C"
