// Launch configuration of the layer's stages (see stages.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>

#include "gemm_fp8.cuh"
#include "gemm_tc.cuh"
#include "kernels.cuh"
#include "stages.cuh"

namespace moe {
namespace stage {

Layout layout(const moe_config& c) {
  const size_t T = c.T, K = c.K, E = c.E, d = c.d, I = c.I, S = c.S;
  const size_t TK = T * K;
  const size_t nch = (size_t)permute_chunks(c.T);
  const bool f8 = is_f8(c.expert);
  const size_t ea = elem_bytes(c.act), ex = elem_bytes(c.expert);
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += align256(bytes);
    return at;
  };
  L.err = take(256);
  L.scores = take(T * E * 4);
  L.local_rank = take(TK * 4);
  L.chunk_hist = take(E * nch * 4);
  L.chunk_base = take(E * nch * 4);
  L.offsets = take((E + 1) * 4);
  const size_t ER = (size_t)expert_rows(c);  // T * K, plus the padding rows of the padded layout
  L.sorted_tok = take(ER * 4);                 // indexed by row position
  L.slot_pos = take(TK * 4);
  const size_t pairs = c.act == MOE_F32 ? 2 : 1;  // fp32 GEMM operands are stored as tf32 pairs
  L.xp = take(ER * d * ex * pairs);
  L.xp_scale = take(f8 ? (d / 128) * TK * 4 : 0);
  L.xq = take(f8 ? T * d : 0);
  L.xq_scale = take(f8 ? (d / 128) * T * 4 : 0);
  L.tok_scale = take(f8 ? (d / 128) * T * 4 : 0);
  L.h = take(ER * I * ex * pairs);
  L.h_scale = take(f8 ? (I / 128) * TK * 4 : 0);
  L.hs = take(T * S * I * ex * pairs);
  L.hs_scale = take(f8 ? (S * I / 128) * T * 4 : 0);
  const bool scat = scatter_combine(c);
  L.yp = take(scat ? 0 : ER * d * ea);
  L.gate_p = take(scat ? ER * 4 : 0);
  L.acc = take(scat && c.act == MOE_BF16 ? T * d * 4 : 0);  // fp32 layers add into out itself
  const bool f32 = c.act == MOE_F32;
  L.xs = take(f32 ? T * 2 * d * 4 : 0);
  L.wr_s = take(f32 ? E * 2 * d * 4 : 0);
  L.w13_s = take(f32 ? E * 2 * I * 2 * d * 4 : 0);
  L.w2_s = take(f32 ? E * d * 2 * I * 4 : 0);
  L.ws13_s = take(f32 ? S * 2 * I * 2 * d * 4 : 0);
  L.ws2_s = take(f32 ? S * d * 2 * I * 4 : 0);
  L.total = o;
  return L;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// ------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Row-major [outer, inner] matrix of `elem`-byte values, box [box_outer, box_inner],
// 128-byte swizzle (box_inner * elem must be 128).
static moe_status map_2d(CUtensorMap* m, const void* ptr, size_t elem, uint64_t inner, uint64_t outer,
                         uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return MOE_ERR_CUDA;
  const CUtensorMapDataType dt = elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * elem};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// [n_mat, outer, inner] stack of matrices, box [1, box_outer, box_inner].
static moe_status map_3d(CUtensorMap* m, const void* ptr, size_t elem, uint64_t inner, uint64_t outer,
                         uint64_t n_mat, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr) return MOE_ERR_CUDA;
  const CUtensorMapDataType dt = elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[3] = {inner, outer, n_mat};
  cuuint64_t strides[2] = {inner * elem, inner * outer * elem};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// fp32 tf32 pairs: [n_mat,] rows, 2, K (K innermost), box [1,] box_rows, 1, 32
// (one 128-byte swizzle row of 32 fp32 per row and part). n_mat = 0: 3-D.
static moe_status map_pairs(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, uint64_t n_mat,
                            uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return MOE_ERR_CUDA;
  const int rank = n_mat ? 4 : 3;
  cuuint64_t dims[4] = {K, 2, rows, n_mat ? n_mat : 1};
  cuuint64_t strides[3] = {K * 4, 2 * K * 4, rows * 2 * K * 4};
  cuuint32_t box[4] = {32, 1, box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_INVALID_ARG;
}

static int down_bn(int d) { return d % 256 == 0 ? 256 : 128; }

// 128-row halves per tile of the bf16 expert GEMMs: 1 by default;
// MOE_GEMM_TILE_ROWS=256 selects 256-row tiles whose two halves share each
// staged weight slice (a third less operand traffic from L2, but a single
// TMEM accumulator, so the epilogue no longer overlaps the next tile's main
// loop; measured slower on every workload here). Read once per process; the
// two tilings give bit-identical results.
static int expert_tile_halves() {
  static int mh = 0;
  if (mh == 0) {
    const char* v = getenv("MOE_GEMM_TILE_ROWS");
    mh = (v != nullptr && atoi(v) == 256) ? 2 : 1;
  }
  return mh;
}

static int router_bn(int E) { return E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256; }

static int tc_grid(long long tiles_upper) {
  return (int)std::max(1LL, std::min((long long)num_sms(), tiles_upper));
}

// ------------------------------------------------------------ stages
// The router GEMM with the sigmoid in its epilogue.
static moe_status router_gemm(const moe_config& c, const void* x, const void* w_router, float* s, void* ws,
                              cudaStream_t st) {
  TcGemmLaunch L{};
  L.epi = Epi::kRouterSigmoid;
  L.bn = router_bn(c.E);
  if (c.act == MOE_F32) {
    // x and w_router as tf32 pairs
    L.split = true;
    MOE_TRY(map_pairs(&L.a1, x, c.d, c.T, 0, 128));
    MOE_TRY(map_pairs(&L.b1, w_router, c.d, c.E, 0, L.bn));
    L.p.k_blocks1 = c.d / 32;
  } else {
    MOE_TRY(map_2d(&L.a1, x, 2, c.d, c.T, 64, 128));
    MOE_TRY(map_2d(&L.b1, w_router, 2, c.d, c.E, 64, L.bn));
    L.p.k_blocks1 = c.d / 64;
  }
  L.a0 = L.a1;
  L.b0 = L.b1;
  L.p.groups0 = 0;
  L.p.rows1 = c.T;
  L.p.n_tiles1 = (c.E + L.bn - 1) / L.bn;  // more than one only past 256 experts (fp32 layers)
  L.p.out1 = s;
  L.p.n_valid = c.E;
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid((long long)((c.T + 127) / 128) * L.p.n_tiles1);
  L.stream = st;
  MOE_CUDA(launch_tc_gemm(L));
  return MOE_OK;
}

moe_status router_scores(const moe_config& c, const void* x, const void* w_router, float* s, void* ws,
                         cudaStream_t st) {
  return router_gemm(c, x, w_router, s, ws, st);
}

F32W f32_weights(const moe_config& c, void* ws) {
  const Layout L = layout(c);
  return F32W{at<float>(ws, L.wr_s), at<float>(ws, L.w13_s), at<float>(ws, L.w2_s), at<float>(ws, L.ws13_s),
              at<float>(ws, L.ws2_s)};
}

moe_status split_rows_f32(const void* src, long long rows, int cols, void* dst, cudaStream_t st) {
  MOE_CUDA(launch_split_tf32(static_cast<const float*>(src), rows, cols, static_cast<float*>(dst), num_sms(), st));
  return MOE_OK;
}

moe_status split_weights_f32(const moe_config& c, const moe_weights* w, bool router, bool routed, bool shared,
                             void* ws, cudaStream_t st) {
  const F32W f = f32_weights(c, ws);
  if (router) MOE_TRY(split_rows_f32(w->w_router, c.E, c.d, f.wr, st));
  if (routed) {
    MOE_TRY(split_rows_f32(w->w13, (long long)c.E * 2 * c.I, c.d, f.w13, st));
    MOE_TRY(split_rows_f32(w->w2, (long long)c.E * c.d, c.I, f.w2, st));
  }
  if (shared && c.S > 0) {
    MOE_TRY(split_rows_f32(w->ws13, (long long)c.S * 2 * c.I, c.d, f.ws13, st));
    MOE_TRY(split_rows_f32(w->ws2, (long long)c.S * c.d, c.I, f.ws2, st));
  }
  return MOE_OK;
}

moe_status route_stage(const moe_config& c, const void* x, const void* w_router, const float* scores_in,
                       const float* bias, float* scores_out, int32_t* topk_idx, float* topk_gate, int32_t* counts,
                       void* ws, cudaStream_t st) {
  MOE_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, st));
  if (c.T == 0) return MOE_OK;
  const float* s = scores_in;
  if (s == nullptr) {
    float* buf = scores_out ? scores_out : at<float>(ws, layout(c).scores);
    if (c.act == MOE_F32) {
      // fp32 router on the tensor cores: x and w_router as tf32 pairs
      void* xs = at<void>(ws, layout(c).xs);
      MOE_TRY(split_rows_f32(x, c.T, c.d, xs, st));
      MOE_TRY(split_rows_f32(w_router, c.E, c.d, f32_weights(c, ws).wr, st));
      x = xs;
      w_router = f32_weights(c, ws).wr;
    }
    MOE_TRY(router_scores(c, x, w_router, buf, ws, st));
    s = buf;
  } else if (scores_out != nullptr && scores_out != scores_in) {
    MOE_CUDA(cudaMemcpyAsync(scores_out, scores_in, sizeof(float) * c.T * c.E, cudaMemcpyDeviceToDevice, st));
  }
  MOE_CUDA(launch_route_select(s, bias, c.T, c.E, c.G, c.K, c.M, c.group_topk, topk_idx, topk_gate, counts,
                               num_sms(), st));
  return MOE_OK;
}

moe_status permute_stage(const moe_config& c, const int32_t* topk_idx, const int32_t* counts, int32_t* offsets,
                         int32_t* sorted_tok, int32_t* slot_pos, const void* x, void* xp, float* xp_scale,
                         uint8_t* xq, float* xq_scale, void* ws, cudaStream_t st, const float* gate,
                         float* gate_p, bool pairs, int pad) {
  const Layout Lw = layout(c);
  if (c.T == 0) {
    MOE_CUDA(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1), st));
    return MOE_OK;
  }
  int* err = at<int>(ws, 0);
  int* local_rank = at<int>(ws, Lw.local_rank);
  int* chunk_hist = at<int>(ws, Lw.chunk_hist);
  int* chunk_base = at<int>(ws, Lw.chunk_base);
  MOE_CUDA(launch_permute_rank(topk_idx, c.T, c.K, c.E, local_rank, chunk_hist, err, st));
  MOE_CUDA(launch_permute_scan(counts, chunk_hist, c.T, c.E, chunk_base, offsets, err, st, pad));
  if (is_f8(c.expert)) {
    MOE_CUDA(launch_permute_scatter_e4m3(topk_idx, local_rank, chunk_base, c.T, c.K, c.E,
                                         static_cast<const __nv_bfloat16*>(x), c.d, sorted_tok, slot_pos,
                                         static_cast<uint8_t*>(xp), xp_scale, xq, xq_scale,
                                         at<float>(ws, Lw.tok_scale), c.expert == MOE_E4M3_UE8M0, num_sms(), st,
                                         gate, gate_p));
  } else {
    MOE_CUDA(launch_permute_scatter(topk_idx, local_rank, chunk_base, c.T, c.K, c.E, x,
                                    (size_t)c.d * elem_bytes(c.act) * (pairs ? 2 : 1), sorted_tok, slot_pos, xp,
                                    num_sms(), st, gate, gate_p, pad, offsets, counts));
  }
  return MOE_OK;
}

// ---- FP8 expert GEMMs (e4m3 tiles; fp32 promotion per 128-wide K block, or
// tensor-core block scaling for power-of-two scales)
static cudaError_t launch_f8(const moe_config& c, const Fp8GemmLaunch& L) {
  return c.expert == MOE_E4M3_UE8M0 ? launch_mx_gemm(L) : launch_fp8_gemm(L);
}

static moe_status fp8_gemm1(const moe_config& c, const void* xp, const float* xp_scale, const int32_t* offsets,
                            const uint8_t* xq, const float* xq_scale, const moe_weights* w, bool routed,
                            bool shared, void* ws, cudaStream_t st) {
  const Layout Lw = layout(c);
  const int TK = c.T * c.K;
  Fp8GemmLaunch L{};
  L.epi = Fp8Epi::kSwiGLU;
  long long tiles = 0;
  if (routed) {
    MOE_TRY(map_2d(&L.a0, xp, 1, c.d, TK, 128, 128));
    MOE_TRY(map_3d(&L.b0, w->w13, 1, c.d, 2 * (uint64_t)c.I, c.E, 128, 64));
    L.p.groups0 = c.E;
    L.p.offsets0 = offsets;
    L.p.rows_total0 = TK;
    L.p.n_tiles0 = c.I / 128;
    L.p.k_blocks0 = c.d / 128;
    L.p.a_scale0 = xp_scale;
    L.p.b_scale0 = w->w13_scale;
    L.p.out0 = at<void>(ws, Lw.h);
    L.p.out_scale0 = at<float>(ws, Lw.h_scale);
    L.p.ldo0 = c.I;
    tiles += ((long long)TK / 128 + c.E) * L.p.n_tiles0;
  }
  if (shared && c.S > 0) {
    MOE_TRY(map_2d(&L.a1, xq, 1, c.d, c.T, 128, 128));
    MOE_TRY(map_3d(&L.b1, w->ws13, 1, c.d, 2 * (uint64_t)c.I, c.S, 128, 64));
    L.p.rows1 = c.T;
    L.p.n_tiles1 = c.S * c.I / 128;
    L.p.k_blocks1 = c.d / 128;
    L.p.a_scale1 = xq_scale;
    L.p.b_scale1 = w->ws13_scale;
    L.p.out1 = at<void>(ws, Lw.hs);
    L.p.out_scale1 = at<float>(ws, Lw.hs_scale);
    L.p.ldo1 = c.S * c.I;
    tiles += (long long)((c.T + 127) / 128) * L.p.n_tiles1;
  }
  if (tiles == 0) return MOE_OK;
  if (!routed) {
    L.a0 = L.a1;
    L.b0 = L.b1;
  }
  if (!(shared && c.S > 0)) {
    L.a1 = L.a0;
    L.b1 = L.b0;
  }
  L.p.I = c.I;
  L.p.N = c.d;
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid(tiles);
  L.stream = st;
  MOE_CUDA(launch_f8(c, L));
  return MOE_OK;
}

static moe_status fp8_gemm2(const moe_config& c, const int32_t* offsets, const moe_weights* w, void* yp,
                            bool shared, const void* radd, void* out, void* ws, cudaStream_t st) {
  const Layout Lw = layout(c);
  const int TK = c.T * c.K;
  Fp8GemmLaunch L{};
  if (!shared) {
    L.epi = Fp8Epi::kStore;
    MOE_TRY(map_2d(&L.a0, at<void>(ws, Lw.h), 1, c.I, TK, 128, 128));
    MOE_TRY(map_3d(&L.b0, w->w2, 1, c.I, c.d, c.E, 128, 256));
    L.a1 = L.a0;
    L.b1 = L.b0;
    L.p.groups0 = c.E;
    L.p.offsets0 = offsets;
    L.p.rows_total0 = TK;
    L.p.n_tiles0 = c.d / 256;
    L.p.k_blocks0 = c.I / 128;
    L.p.a_scale0 = at<float>(ws, Lw.h_scale);
    L.p.b_scale0 = w->w2_scale;
    L.p.out0 = yp;
    L.p.ldo0 = c.d;
    L.grid = tc_grid(((long long)TK / 128 + c.E) * L.p.n_tiles0);
  } else {
    L.epi = Fp8Epi::kCombine;
    MOE_TRY(map_2d(&L.a1, at<void>(ws, Lw.hs), 1, (uint64_t)c.S * c.I, c.T, 128, 128));
    MOE_TRY(map_3d(&L.b1, w->ws2, 1, c.I, c.d, c.S, 128, 256));
    L.a0 = L.a1;
    L.b0 = L.b1;
    L.p.groups0 = 0;
    L.p.rows1 = c.T;
    L.p.n_tiles1 = c.d / 256;
    L.p.k_blocks1 = c.S * c.I / 128;
    L.p.a_scale1 = at<float>(ws, Lw.hs_scale);
    L.p.b_scale1 = w->ws2_scale;
    L.p.out1 = out;
    L.p.ldo1 = c.d;
    L.p.radd = static_cast<const __nv_bfloat16*>(radd);
    L.grid = tc_grid((long long)((c.T + 127) / 128) * L.p.n_tiles1);
  }
  L.p.I = c.I;
  L.p.N = c.d;
  L.p.err = at<int>(ws, 0);
  L.stream = st;
  MOE_CUDA(launch_f8(c, L));
  return MOE_OK;
}

// GEMM1 (SwiGLU) of the routed experts over xp and/or the shared experts over x.
moe_status gemm1_stage(const moe_config& c, const void* xp, const float* xp_scale, const int32_t* offsets,
                       const void* x, const moe_weights* w, bool routed, bool shared, void* ws, cudaStream_t st,
                       int rows) {
  const Layout Lw = layout(c);
  const int TK = rows < 0 ? c.T * c.K : rows;
  if (is_f8(c.expert)) {
    return fp8_gemm1(c, xp, xp_scale, offsets, at<uint8_t>(ws, Lw.xq), at<float>(ws, Lw.xq_scale), w, routed,
                     shared, ws, st);
  }
  // fp32 layers: xp, x and the weights are tf32 pairs (xp and x in the
  // workspace, the weights from split_weights_f32)
  const bool f32 = c.act == MOE_F32;
  const F32W f = f32_weights(c, ws);
  TcGemmLaunch L{};
  L.epi = Epi::kSwiGLU;
  L.mh = expert_tile_halves();
  L.split = f32;
  L.bn = 256;
  const int kbs = f32 ? c.d / 32 : c.d / 64;
  long long tiles = 0;
  if (routed) {
    if (f32) {
      MOE_TRY(map_pairs(&L.a0, xp, c.d, TK, 0, 128));
      MOE_TRY(map_pairs(&L.b0, f.w13, c.d, 2 * (uint64_t)c.I, c.E, 64));
    } else {
      MOE_TRY(map_2d(&L.a0, xp, 2, c.d, TK, 64, 128));
      MOE_TRY(map_3d(&L.b0, w->w13, 2, c.d, 2 * (uint64_t)c.I, c.E, 64, 64));
    }
    L.p.groups0 = c.E;
    L.p.offsets0 = offsets;
    L.p.n_tiles0 = c.I / 128;
    L.p.k_blocks0 = kbs;
    L.p.out0 = at<void>(ws, Lw.h);
    L.p.ldo0 = c.I;
    tiles += ((long long)TK / 128 + c.E) * L.p.n_tiles0;
  }
  if (shared && c.S > 0) {
    if (f32) {
      MOE_TRY(map_pairs(&L.a1, x, c.d, c.T, 0, 128));
      MOE_TRY(map_pairs(&L.b1, f.ws13, c.d, 2 * (uint64_t)c.I, c.S, 64));
    } else {
      MOE_TRY(map_2d(&L.a1, x, 2, c.d, c.T, 64, 128));
      MOE_TRY(map_3d(&L.b1, w->ws13, 2, c.d, 2 * (uint64_t)c.I, c.S, 64, 64));
    }
    L.p.rows1 = c.T;
    L.p.n_tiles1 = c.S * c.I / 128;
    L.p.k_blocks1 = kbs;
    L.p.out1 = at<void>(ws, Lw.hs);
    L.p.ldo1 = c.S * c.I;
    tiles += (long long)((c.T + 127) / 128) * L.p.n_tiles1;
  }
  if (tiles == 0) return MOE_OK;
  if (!routed) {
    L.a0 = L.a1;
    L.b0 = L.b1;
  }
  if (!(shared && c.S > 0)) {
    L.a1 = L.a0;
    L.b1 = L.b0;
  }
  L.p.I = c.I;
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid(tiles);
  L.stream = st;
  MOE_CUDA(launch_tc_gemm(L));
  return MOE_OK;
}

// Operand maps of a down projection into segment 0 (routed) or 1 (shared):
// A = h [rows, hk] (fp32 layers: tf32 pairs [rows, 2, hk]), B = the W2 stack
// [n_mat, d, I] (fp32 layers: its split copy w2s [n_mat, d, 2, I]).
static moe_status down_maps(const moe_config& c, TcGemmLaunch& L, bool seg1, const void* h, uint64_t hk,
                            uint64_t rows, const void* w2, const float* w2s, uint64_t n_mat) {
  CUtensorMap* a = seg1 ? &L.a1 : &L.a0;
  CUtensorMap* b = seg1 ? &L.b1 : &L.b0;
  const bool f32 = c.act == MOE_F32;
  L.split = f32;
  if (f32) {
    MOE_TRY(map_pairs(a, h, hk, rows, 0, 128));
    MOE_TRY(map_pairs(b, w2s, c.I, c.d, n_mat, L.bn));
  } else {
    MOE_TRY(map_2d(a, h, 2, hk, rows, 64, 128));
    MOE_TRY(map_3d(b, w2, 2, c.I, c.d, n_mat, 64, L.bn));
  }
  const int kb = (int)(hk / (f32 ? 32 : 64));
  if (seg1) {
    L.p.k_blocks1 = kb;
    L.a0 = L.a1;
    L.b0 = L.b1;
  } else {
    L.p.k_blocks0 = kb;
    L.a1 = L.a0;
    L.b1 = L.b0;
  }
  return MOE_OK;
}

// GEMM2 of the routed experts: yp = h W2^T (not gate-scaled).
moe_status gemm2_routed_stage(const moe_config& c, const int32_t* offsets, const moe_weights* w, void* yp, void* ws,
                              cudaStream_t st, int rows, const int32_t* counts) {
  const Layout Lw = layout(c);
  const int TK = rows < 0 ? c.T * c.K : rows;
  if (is_f8(c.expert)) return fp8_gemm2(c, offsets, w, yp, false, nullptr, nullptr, ws, st);
  TcGemmLaunch L{};
  L.epi = c.act == MOE_F32 ? Epi::kStoreF32 : Epi::kStore;
  L.mh = expert_tile_halves();
  L.bn = down_bn(c.d);
  MOE_TRY(down_maps(c, L, false, at<void>(ws, Lw.h), c.I, TK, w->w2, f32_weights(c, ws).w2, c.E));
  L.p.groups0 = c.E;
  L.p.offsets0 = offsets;
  L.p.counts0 = counts;
  L.p.n_tiles0 = c.d / L.bn;
  L.p.out0 = yp;
  L.p.ldo0 = c.d;
  L.p.I = c.I;
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid(((long long)TK / 128 + c.E) * L.p.n_tiles0);
  L.stream = st;
  MOE_CUDA(launch_tc_gemm(L));
  return MOE_OK;
}

moe_status shared_seed_stage(const moe_config& c, const moe_weights* w, float* acc, void* ws, cudaStream_t st) {
  if (c.S == 0) {
    MOE_CUDA(cudaMemsetAsync(acc, 0, sizeof(float) * (size_t)c.T * c.d, st));
    return MOE_OK;
  }
  const Layout Lw = layout(c);
  TcGemmLaunch L{};
  L.epi = Epi::kStoreF32;
  L.mh = expert_tile_halves();
  L.bn = down_bn(c.d);
  MOE_TRY(down_maps(c, L, true, at<void>(ws, Lw.hs), (uint64_t)c.S * c.I, c.T, w->ws2, f32_weights(c, ws).ws2,
                    c.S));
  L.p.groups0 = 0;
  L.p.rows1 = c.T;
  L.p.n_tiles1 = c.d / L.bn;
  L.p.out1 = acc;
  L.p.ldo1 = c.d;
  L.p.I = c.I;
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid((long long)((c.T + 127) / 128) * L.p.n_tiles1);
  L.stream = st;
  MOE_CUDA(launch_tc_gemm(L));
  return MOE_OK;
}

moe_status gemm2_scatter_stage(const moe_config& c, const int32_t* offsets, const moe_weights* w, float* acc,
                               void* ws, cudaStream_t st) {
  const Layout Lw = layout(c);
  const int TK = c.T * c.K;
  TcGemmLaunch L{};
  L.epi = Epi::kScatterAdd;
  L.mh = expert_tile_halves();
  L.bn = down_bn(c.d);
  MOE_TRY(down_maps(c, L, false, at<void>(ws, Lw.h), c.I, TK, w->w2, f32_weights(c, ws).w2, c.E));
  L.p.groups0 = c.E;
  L.p.offsets0 = offsets;
  L.p.n_tiles0 = c.d / L.bn;
  L.p.out0 = acc;
  L.p.ldo0 = c.d;
  L.p.I = c.I;
  L.p.sorted_tok = at<int>(ws, Lw.sorted_tok);
  L.p.gate_p = at<float>(ws, Lw.gate_p);
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid(((long long)TK / 128 + c.E) * L.p.n_tiles0);
  L.stream = st;
  MOE_CUDA(launch_tc_gemm(L));
  return MOE_OK;
}

moe_status acc_round_stage(const moe_config& c, const float* acc, void* out, cudaStream_t st) {
  MOE_CUDA(launch_acc_to_bf16(acc, (size_t)c.T * c.d, out, num_sms(), st));
  return MOE_OK;
}

// Shared experts' down projection with the gate-weighted routed rows added in
// its epilogue (or a plain gather-sum when there are no shared experts).
moe_status gemm2_combine_stage(const moe_config& c, const void* yp, const int32_t* slot_pos, const float* gate,
                               const moe_weights* w, void* out, void* ws, cudaStream_t st) {
  const Layout Lw = layout(c);
  const bool f32 = c.act == MOE_F32;
  if (c.S == 0) {
    if (f32) {
      MOE_CUDA(launch_gather_combine(yp, slot_pos, gate, c.T, c.d, c.K, false, out, num_sms(), st));
    } else {
      MOE_CUDA(launch_routed_sum_bf16(yp, slot_pos, gate, c.T, c.d, c.K, out, num_sms(), st));
    }
    return MOE_OK;
  }
  // routed sum r[t] (in the xp region of the workspace: the permuted rows are
  // dead once the routed GEMM1 has run), added by the down projection's epilogue
  void* r = at<void>(ws, Lw.xp);
  if (f32) {
    MOE_CUDA(launch_gather_combine(yp, slot_pos, gate, c.T, c.d, c.K, false, r, num_sms(), st));
  } else {
    MOE_CUDA(launch_routed_sum_bf16(yp, slot_pos, gate, c.T, c.d, c.K, r, num_sms(), st));
  }
  if (is_f8(c.expert)) return fp8_gemm2(c, nullptr, w, nullptr, true, r, out, ws, st);
  TcGemmLaunch L{};
  L.epi = Epi::kCombine;
  L.mh = expert_tile_halves();
  L.bn = down_bn(c.d);
  MOE_TRY(down_maps(c, L, true, at<void>(ws, Lw.hs), (uint64_t)c.S * c.I, c.T, w->ws2, f32_weights(c, ws).ws2,
                    c.S));
  L.p.groups0 = 0;
  L.p.rows1 = c.T;
  L.p.n_tiles1 = c.d / L.bn;
  L.p.out1 = out;
  L.p.ldo1 = c.d;
  L.p.I = c.I;
  L.p.radd = static_cast<const __nv_bfloat16*>(r);
  L.p.radd_f32 = static_cast<const float*>(r);
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid((long long)((c.T + 127) / 128) * L.p.n_tiles1);
  L.stream = st;
  MOE_CUDA(launch_tc_gemm(L));
  return MOE_OK;
}

}  // namespace stage
}  // namespace moe
