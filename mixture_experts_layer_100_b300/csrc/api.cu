// C ABI of the MoE layer library: argument checks, workspace layout, TMA
// tensor maps and the launch sequence of each entry point (see moe.h).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "gemm_fp8.cuh"
#include "gemm_tc.cuh"
#include "kernels.cuh"
#include "moe.h"

using namespace moe;

namespace {

#define MOE_CUDA(call)                              \
  do {                                              \
    cudaError_t e_ = (call);                        \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA;     \
  } while (0)

#define MOE_TRY(call)                   \
  do {                                  \
    moe_status s_ = (call);             \
    if (s_ != MOE_OK) return s_;        \
  } while (0)

size_t elem_bytes(moe_dtype t) { return t == MOE_F32 ? 4 : t == MOE_BF16 ? 2 : 1; }

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_f8(moe_dtype t) { return t == MOE_E4M3 || t == MOE_E4M3_UE8M0; }

// ------------------------------------------------------------ workspace
struct Layout {
  size_t err, scores, local_rank, chunk_hist, chunk_base, offsets, sorted_tok, slot_pos;
  size_t xp, xp_scale, xq, xq_scale, tok_scale, h, h_scale, hs, hs_scale, yp, total;
};

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
  L.sorted_tok = take(TK * 4);
  L.slot_pos = take(TK * 4);
  L.xp = take(TK * d * ex);
  L.xp_scale = take(f8 ? (d / 128) * TK * 4 : 0);
  L.xq = take(f8 ? T * d : 0);
  L.xq_scale = take(f8 ? (d / 128) * T * 4 : 0);
  L.tok_scale = take(f8 ? (d / 128) * T * 4 : 0);
  L.h = take(TK * I * ex);
  L.h_scale = take(f8 ? (I / 128) * TK * 4 : 0);
  L.hs = take(T * S * I * ex);
  L.hs_scale = take(f8 ? (S * I / 128) * T * 4 : 0);
  L.yp = take(TK * d * ea);
  L.total = o;
  return L;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

// ------------------------------------------------------------ checks
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
  if (c->act == MOE_BF16) {
    if (c->d % 128 != 0 || c->I % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (c->E > 256) return MOE_ERR_UNSUPPORTED;
    if (is_f8(c->expert) && c->d % 256 != 0) return MOE_ERR_UNSUPPORTED;
  } else if (c->d % 4 != 0) {
    return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
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
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
moe_status map_2d(CUtensorMap* m, const void* ptr, size_t elem, uint64_t inner, uint64_t outer, uint32_t box_inner,
                  uint32_t box_outer) {
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
moe_status map_3d(CUtensorMap* m, const void* ptr, size_t elem, uint64_t inner, uint64_t outer, uint64_t n_mat,
                  uint32_t box_inner, uint32_t box_outer) {
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

int down_bn(int d) { return d % 256 == 0 ? 256 : 128; }

int router_bn(int E) { return E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256; }

int tc_grid(long long tiles_upper) {
  return (int)std::max(1LL, std::min((long long)num_sms(), tiles_upper));
}

// ------------------------------------------------------------ stages
moe_status router_scores(const moe_config& c, const void* x, const void* w_router, float* s, void* ws,
                         cudaStream_t st) {
  if (c.act == MOE_F32) {
    MOE_CUDA(launch_router_f32(static_cast<const float*>(x), static_cast<const float*>(w_router), c.T, c.d, c.E, s,
                               st));
    return MOE_OK;
  }
  TcGemmLaunch L{};
  L.epi = Epi::kRouterSigmoid;
  L.bn = router_bn(c.E);
  MOE_TRY(map_2d(&L.a1, x, 2, c.d, c.T, 64, 128));
  MOE_TRY(map_2d(&L.b1, w_router, 2, c.d, c.E, 64, L.bn));
  L.a0 = L.a1;
  L.b0 = L.b1;
  L.p.groups0 = 0;
  L.p.rows1 = c.T;
  L.p.n_tiles1 = 1;
  L.p.k_blocks1 = c.d / 64;
  L.p.out1 = s;
  L.p.n_valid = c.E;
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid((c.T + 127) / 128);
  L.stream = st;
  MOE_CUDA(launch_tc_gemm(L));
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
                         uint8_t* xq, float* xq_scale, void* ws, cudaStream_t st) {
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
  MOE_CUDA(launch_permute_scan(counts, chunk_hist, c.T, c.E, chunk_base, offsets, err, st));
  if (is_f8(c.expert)) {
    MOE_CUDA(launch_permute_scatter_e4m3(topk_idx, local_rank, chunk_base, c.T, c.K, c.E,
                                         static_cast<const __nv_bfloat16*>(x), c.d, sorted_tok, slot_pos,
                                         static_cast<uint8_t*>(xp), xp_scale, xq, xq_scale,
                                         at<float>(ws, Lw.tok_scale), c.expert == MOE_E4M3_UE8M0, num_sms(), st));
  } else {
    MOE_CUDA(launch_permute_scatter(topk_idx, local_rank, chunk_base, c.T, c.K, c.E, x, (size_t)c.d * elem_bytes(c.act),
                                    sorted_tok, slot_pos, xp, num_sms(), st));
  }
  return MOE_OK;
}

// ---- FP8 expert GEMMs (e4m3 tiles; fp32 promotion per 128-wide K block, or
// tensor-core block scaling for power-of-two scales)
cudaError_t launch_f8(const moe_config& c, const Fp8GemmLaunch& L) {
  return c.expert == MOE_E4M3_UE8M0 ? launch_mx_gemm(L) : launch_fp8_gemm(L);
}

moe_status fp8_gemm1(const moe_config& c, const void* xp, const float* xp_scale, const int32_t* offsets,
                     const uint8_t* xq, const float* xq_scale, const moe_weights* w, bool routed, bool shared,
                     void* ws, cudaStream_t st) {
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

moe_status fp8_gemm2(const moe_config& c, const int32_t* offsets, const moe_weights* w, void* yp, bool shared,
                     const void* radd, void* out, void* ws, cudaStream_t st) {
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
                       const void* x, const moe_weights* w, bool routed, bool shared, void* ws, cudaStream_t st) {
  const Layout Lw = layout(c);
  const int TK = c.T * c.K;
  if (c.act == MOE_F32) {
    if (routed) {
      SimtParams p{};
      p.mode = kSimtSwiGLU;
      p.A = static_cast<const float*>(xp);
      p.lda = c.d;
      p.B = static_cast<const float*>(w->w13);
      p.groups = c.E;
      p.offsets = offsets;
      p.N = c.I;
      p.Kdim = c.d;
      p.I = c.I;
      p.out = at<float>(ws, Lw.h);
      p.ldo = c.I;
      MOE_CUDA(launch_simt_gemm(p, simt_max_mtiles(TK, c.E), st));
    }
    if (shared && c.S > 0) {
      SimtParams p{};
      p.mode = kSimtSwiGLU;
      p.A = static_cast<const float*>(x);
      p.lda = c.d;
      p.B = static_cast<const float*>(w->ws13);
      p.rows = c.T;
      p.shared = 1;
      p.N = c.S * c.I;
      p.Kdim = c.d;
      p.I = c.I;
      p.out = at<float>(ws, Lw.hs);
      p.ldo = c.S * c.I;
      MOE_CUDA(launch_simt_gemm(p, simt_max_mtiles(c.T, 0), st));
    }
    return MOE_OK;
  }
  if (is_f8(c.expert)) {
    return fp8_gemm1(c, xp, xp_scale, offsets, at<uint8_t>(ws, Lw.xq), at<float>(ws, Lw.xq_scale), w, routed,
                     shared, ws, st);
  }
  TcGemmLaunch L{};
  L.epi = Epi::kSwiGLU;
  L.bn = 256;
  long long tiles = 0;
  if (routed) {
    MOE_TRY(map_2d(&L.a0, xp, 2, c.d, TK, 64, 128));
    MOE_TRY(map_3d(&L.b0, w->w13, 2, c.d, 2 * (uint64_t)c.I, c.E, 64, 64));
    L.p.groups0 = c.E;
    L.p.offsets0 = offsets;
    L.p.n_tiles0 = c.I / 128;
    L.p.k_blocks0 = c.d / 64;
    L.p.out0 = at<void>(ws, Lw.h);
    L.p.ldo0 = c.I;
    tiles += ((long long)TK / 128 + c.E) * L.p.n_tiles0;
  }
  if (shared && c.S > 0) {
    MOE_TRY(map_2d(&L.a1, x, 2, c.d, c.T, 64, 128));
    MOE_TRY(map_3d(&L.b1, w->ws13, 2, c.d, 2 * (uint64_t)c.I, c.S, 64, 64));
    L.p.rows1 = c.T;
    L.p.n_tiles1 = c.S * c.I / 128;
    L.p.k_blocks1 = c.d / 64;
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

// GEMM2 of the routed experts: yp = h W2^T (not gate-scaled).
moe_status gemm2_routed_stage(const moe_config& c, const int32_t* offsets, const moe_weights* w, void* yp, void* ws,
                              cudaStream_t st) {
  const Layout Lw = layout(c);
  const int TK = c.T * c.K;
  if (c.act == MOE_F32) {
    SimtParams p{};
    p.mode = kSimtStore;
    p.A = at<float>(ws, Lw.h);
    p.lda = c.I;
    p.B = static_cast<const float*>(w->w2);
    p.groups = c.E;
    p.offsets = offsets;
    p.N = c.d;
    p.Kdim = c.I;
    p.I = c.I;
    p.out = static_cast<float*>(yp);
    p.ldo = c.d;
    MOE_CUDA(launch_simt_gemm(p, simt_max_mtiles(TK, c.E), st));
    return MOE_OK;
  }
  if (is_f8(c.expert)) return fp8_gemm2(c, offsets, w, yp, false, nullptr, nullptr, ws, st);
  TcGemmLaunch L{};
  L.epi = Epi::kStore;
  L.bn = down_bn(c.d);
  MOE_TRY(map_2d(&L.a0, at<void>(ws, Lw.h), 2, c.I, TK, 64, 128));
  MOE_TRY(map_3d(&L.b0, w->w2, 2, c.I, c.d, c.E, 64, L.bn));
  L.a1 = L.a0;
  L.b1 = L.b0;
  L.p.groups0 = c.E;
  L.p.offsets0 = offsets;
  L.p.n_tiles0 = c.d / L.bn;
  L.p.k_blocks0 = c.I / 64;
  L.p.out0 = yp;
  L.p.ldo0 = c.d;
  L.p.I = c.I;
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid(((long long)TK / 128 + c.E) * L.p.n_tiles0);
  L.stream = st;
  MOE_CUDA(launch_tc_gemm(L));
  return MOE_OK;
}

// Shared experts' down projection with the gate-weighted routed rows added in
// its epilogue (or a plain gather-sum when there are no shared experts).
moe_status gemm2_combine_stage(const moe_config& c, const void* yp, const int32_t* slot_pos, const float* gate,
                               const moe_weights* w, void* out, void* ws, cudaStream_t st) {
  const Layout Lw = layout(c);
  if (c.S == 0) {
    if (c.act == MOE_BF16) {
      MOE_CUDA(launch_routed_sum_bf16(yp, slot_pos, gate, c.T, c.d, c.K, out, num_sms(), st));
    } else {
      MOE_CUDA(launch_gather_combine(yp, slot_pos, gate, c.T, c.d, c.K, false, out, num_sms(), st));
    }
    return MOE_OK;
  }
  if (c.act == MOE_F32) {
    SimtParams p{};
    p.mode = kSimtCombine;
    p.A = at<float>(ws, Lw.hs);
    p.lda = c.S * c.I;
    p.B = static_cast<const float*>(w->ws2);
    p.rows = c.T;
    p.shared = 1;
    p.N = c.d;
    p.Kdim = c.S * c.I;
    p.I = c.I;
    p.out = static_cast<float*>(out);
    p.ldo = c.d;
    p.slot_pos = slot_pos;
    p.gate = gate;
    p.yp = static_cast<const float*>(yp);
    p.topk = c.K;
    MOE_CUDA(launch_simt_gemm(p, simt_max_mtiles(c.T, 0), st));
    return MOE_OK;
  }
  // routed sum r[t] (in the xp region of the workspace: the permuted rows are
  // dead once the routed GEMM1 has run), added by the down projection's epilogue
  void* r = at<void>(ws, Lw.xp);
  MOE_CUDA(launch_routed_sum_bf16(yp, slot_pos, gate, c.T, c.d, c.K, r, num_sms(), st));
  if (is_f8(c.expert)) return fp8_gemm2(c, nullptr, w, nullptr, true, r, out, ws, st);
  TcGemmLaunch L{};
  L.epi = Epi::kCombine;
  L.bn = down_bn(c.d);
  MOE_TRY(map_2d(&L.a1, at<void>(ws, Lw.hs), 2, (uint64_t)c.S * c.I, c.T, 64, 128));
  MOE_TRY(map_3d(&L.b1, w->ws2, 2, c.I, c.d, c.S, 64, L.bn));
  L.a0 = L.a1;
  L.b0 = L.b1;
  L.p.groups0 = 0;
  L.p.rows1 = c.T;
  L.p.n_tiles1 = c.d / L.bn;
  L.p.k_blocks1 = c.S * c.I / 64;
  L.p.out1 = out;
  L.p.ldo1 = c.d;
  L.p.I = c.I;
  L.p.radd = static_cast<const __nv_bfloat16*>(r);
  L.p.err = at<int>(ws, 0);
  L.grid = tc_grid((long long)((c.T + 127) / 128) * L.p.n_tiles1);
  L.stream = st;
  MOE_CUDA(launch_tc_gemm(L));
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

moe_status stage_mark(int i, cudaStream_t st) {
  if (g_stage_on) MOE_CUDA(cudaEventRecord(g_stage_events[i], st));
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
  const Layout Lw = layout(c);
  MOE_TRY(stage_mark(0, st));
  MOE_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * c.E, st));
  if (c.T > 0) {
    float* scores = at<float>(ws, Lw.scores);
    const bool f8 = is_f8(c.expert);
    MOE_TRY(router_scores(c, x, w->w_router, scores, ws, st));
    MOE_TRY(stage_mark(1, st));
    // The shared experts' GEMM1 depends on x only: it runs on a side stream,
    // overlapping the memory-bound selection and permutation below; the main
    // stream waits for it before the shared down projection.
    SideStream* side = nullptr;
    if (c.S > 0) {
      MOE_TRY(side_stream(&side));
      MOE_CUDA(cudaEventRecord(side->fork, st));
      MOE_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
      if (f8) {
        MOE_CUDA(launch_quantize_rows(static_cast<const __nv_bfloat16*>(x), c.T, c.d, at<uint8_t>(ws, Lw.xq),
                                      at<float>(ws, Lw.xq_scale), c.expert == MOE_E4M3_UE8M0, num_sms(),
                                      side->s));
      }
      MOE_TRY(gemm1_stage(c, nullptr, nullptr, nullptr, x, w, false, true, ws, side->s));
      MOE_CUDA(cudaEventRecord(side->join, side->s));
    }
    MOE_CUDA(launch_route_select(scores, bias, c.T, c.E, c.G, c.K, c.M, c.group_topk, topk_idx, topk_gate, counts,
                                 num_sms(), st));
    MOE_TRY(stage_mark(2, st));
    int32_t* offsets = at<int32_t>(ws, Lw.offsets);
    int32_t* slot_pos = at<int32_t>(ws, Lw.slot_pos);
    void* xp = at<void>(ws, Lw.xp);
    void* yp = at<void>(ws, Lw.yp);
    MOE_TRY(permute_stage(c, topk_idx, counts, offsets, at<int32_t>(ws, Lw.sorted_tok), slot_pos, x, xp,
                          f8 ? at<float>(ws, Lw.xp_scale) : nullptr, nullptr, nullptr, ws, st));
    MOE_TRY(stage_mark(3, st));
    MOE_TRY(gemm1_stage(c, xp, f8 ? at<float>(ws, Lw.xp_scale) : nullptr, offsets, x, w, true, false, ws, st));
    MOE_TRY(stage_mark(4, st));
    MOE_TRY(gemm2_routed_stage(c, offsets, w, yp, ws, st));
    MOE_TRY(stage_mark(5, st));
    if (side != nullptr) MOE_CUDA(cudaStreamWaitEvent(st, side->join, 0));
    MOE_TRY(gemm2_combine_stage(c, yp, slot_pos, topk_gate, w, out, ws, st));
    MOE_TRY(stage_mark(6, st));
    if (gamma != 0.0f)
      MOE_CUDA(launch_bias_update(counts, c.E, (long long)c.T * c.K, gamma, bias, max_over_mean, st));
    MOE_TRY(stage_mark(7, st));
  }
  return MOE_OK;
}

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

moe_status moe_set_stage_events(void* const* events, int count) {
  if (count == 0) {
    g_stage_on = false;
    return MOE_OK;
  }
  if (events == nullptr || count < 8) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 8; ++i) {
    if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
    g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
  }
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
