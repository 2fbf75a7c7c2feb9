// Launch configuration of the layer's stages: the workspace layout, the TMA
// tensor maps and the kernel launches of each stage. The C ABI (api.cu)
// validates arguments and calls these; the recorded DRAM traffic of the
// GEMM kernels depends on this file and the kernels, not on the ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "moe.h"

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

namespace moe {
namespace stage {

inline size_t elem_bytes(moe_dtype t) { return t == MOE_F32 ? 4 : t == MOE_BF16 ? 2 : 1; }

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool is_f8(moe_dtype t) { return t == MOE_E4M3 || t == MOE_E4M3_UE8M0; }

// moe_layer_forward combines by fp32 reductions in the routed down
// projection's epilogue (bf16 or fp32 layers; not the FP8 expert GEMMs).
inline bool scatter_combine(const moe_config& c) {
  return c.combine == MOE_COMBINE_SCATTER_ADD && c.act == c.expert;
}

// moe_layer_forward's expert-row layout: with bf16 expert GEMMs, the gather
// combine and at least 128 rows per expert on average, every expert's rows
// start at a multiple of 128 and the (at most 127) rows after them are zero,
// so the last tile of each expert multiplies zeros, not the next expert's
// rows (same results, less power under the cap). Other layers, and the
// separate entry points, keep the rows contiguous.
inline bool zero_padded(const moe_config& c) {
  const long long tk = (long long)c.T * c.K;
  return c.act == MOE_BF16 && c.expert == MOE_BF16 && !scatter_combine(c) && tk >= 128LL * c.E &&
         tk + 127LL * c.E <= 0x7fffffffLL;
}
// Rows of the layer's permuted buffers (xp, h, yp).
inline int expert_rows(const moe_config& c) { return c.T * c.K + (zero_padded(c) ? 127 * c.E : 0); }

// ------------------------------------------------------------ workspace
struct Layout {
  size_t err, scores, local_rank, chunk_hist, chunk_base, offsets, sorted_tok, slot_pos;
  size_t xp, xp_scale, xq, xq_scale, tok_scale, h, h_scale, hs, hs_scale, yp, gate_p, acc;
  // fp32 layers: x and the weights as tf32 pairs (see F32W)
  size_t xs, wr_s, w13_s, w2_s, ws13_s, ws2_s;
  size_t total;
};

Layout layout(const moe_config& c);

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

int num_sms();

// ---- fp32 layers: every GEMM operand as tf32 pairs ([rows, 2, K]: the tf32
// high parts of a row, then the remainders), multiplied as hi*hi + hi*lo +
// lo*hi on the tensor cores (kind::tf32, fp32 accumulation).
struct F32W {
  float *wr, *w13, *w2, *ws13, *ws2;  // [E,2,d], [E,2I,2,d], [E,d,2,I], [S,2I,2,d], [S,d,2,I]
};
F32W f32_weights(const moe_config& c, void* ws);
// Splits the weights named by the flags into the workspace.
moe_status split_weights_f32(const moe_config& c, const moe_weights* w, bool router, bool routed, bool shared,
                             void* ws, cudaStream_t st);
// fp32 rows [rows, cols] -> tf32 pairs [rows, 2, cols].
moe_status split_rows_f32(const void* src, long long rows, int cols, void* dst, cudaStream_t st);

// Router GEMM + sigmoid, scores s [T, E]. For fp32 layers x and w_router are
// the tf32 pairs (ws xs, F32W::wr).
moe_status router_scores(const moe_config& c, const void* x, const void* w_router, float* s, void* ws,
                         cudaStream_t st);
moe_status route_stage(const moe_config& c, const void* x, const void* w_router, const float* scores_in,
                       const float* bias, float* scores_out, int32_t* topk_idx, float* topk_gate, int32_t* counts,
                       void* ws, cudaStream_t st);
moe_status permute_stage(const moe_config& c, const int32_t* topk_idx, const int32_t* counts, int32_t* offsets,
                         int32_t* sorted_tok, int32_t* slot_pos, const void* x, void* xp, float* xp_scale,
                         uint8_t* xq, float* xq_scale, void* ws, cudaStream_t st, const float* gate = nullptr,
                         float* gate_p = nullptr, bool pairs = false, int pad = 1);
// rows: rows of xp and of the workspace h (T * K, or expert_rows(c) for the
// padded layout).
moe_status gemm1_stage(const moe_config& c, const void* xp, const float* xp_scale, const int32_t* offsets,
                       const void* x, const moe_weights* w, bool routed, bool shared, void* ws, cudaStream_t st,
                       int rows = -1);
// counts (padded layout): the down projection writes only each expert's own
// rows, not the zero rows after them.
moe_status gemm2_routed_stage(const moe_config& c, const int32_t* offsets, const moe_weights* w, void* yp, void* ws,
                              cudaStream_t st, int rows = -1, const int32_t* counts = nullptr);
// Scatter-add combine: the shared experts' down projection writes the fp32
// accumulator (zeros when S = 0); the routed down projection adds gate * row
// into it; the accumulator is rounded to bf16 out.
moe_status shared_seed_stage(const moe_config& c, const moe_weights* w, float* acc, void* ws, cudaStream_t st);
moe_status gemm2_scatter_stage(const moe_config& c, const int32_t* offsets, const moe_weights* w, float* acc,
                               void* ws, cudaStream_t st);
moe_status acc_round_stage(const moe_config& c, const float* acc, void* out, cudaStream_t st);
moe_status gemm2_combine_stage(const moe_config& c, const void* yp, const int32_t* slot_pos, const float* gate,
                               const moe_weights* w, void* out, void* ws, cudaStream_t st);

}  // namespace stage
}  // namespace moe
