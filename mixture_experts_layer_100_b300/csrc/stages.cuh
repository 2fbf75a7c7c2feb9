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

// ------------------------------------------------------------ workspace
struct Layout {
  size_t err, scores, local_rank, chunk_hist, chunk_base, offsets, sorted_tok, slot_pos;
  size_t xp, xp_scale, xq, xq_scale, tok_scale, h, h_scale, hs, hs_scale, yp, total;
};

Layout layout(const moe_config& c);

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

int num_sms();

moe_status router_scores(const moe_config& c, const void* x, const void* w_router, float* s, void* ws,
                         cudaStream_t st);
moe_status route_stage(const moe_config& c, const void* x, const void* w_router, const float* scores_in,
                       const float* bias, float* scores_out, int32_t* topk_idx, float* topk_gate, int32_t* counts,
                       void* ws, cudaStream_t st);
moe_status permute_stage(const moe_config& c, const int32_t* topk_idx, const int32_t* counts, int32_t* offsets,
                         int32_t* sorted_tok, int32_t* slot_pos, const void* x, void* xp, float* xp_scale,
                         uint8_t* xq, float* xq_scale, void* ws, cudaStream_t st);
moe_status gemm1_stage(const moe_config& c, const void* xp, const float* xp_scale, const int32_t* offsets,
                       const void* x, const moe_weights* w, bool routed, bool shared, void* ws, cudaStream_t st);
moe_status gemm2_routed_stage(const moe_config& c, const int32_t* offsets, const moe_weights* w, void* yp, void* ws,
                              cudaStream_t st);
moe_status gemm2_combine_stage(const moe_config& c, const void* yp, const int32_t* slot_pos, const float* gate,
                               const moe_weights* w, void* out, void* ws, cudaStream_t st);

}  // namespace stage
}  // namespace moe
