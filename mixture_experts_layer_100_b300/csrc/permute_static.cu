// moe_permute_static: the expert-major permutation of moe_permute, for
// callers that cannot allocate device memory (see moe.h). Its scratch space
// is one fixed array in this file instead of a caller-provided workspace.
#include "kernels.cuh"
#include "moe.h"

namespace {

// Scratch of every moe_permute_static call on a device: the device error
// word, per-pair ranks, per-chunk histograms and per-chunk bases. Loading the
// library reserves it on every GPU the process uses, until the process ends.
static __device__ __align__(256) unsigned char g_permute_scratch[MOE_PERMUTE_STATIC_SCRATCH_BYTES];

size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

// Device address of the array in the current context. The host-side name of
// the array is not a device address, so it is asked for on every call: the
// answer then always belongs to the context the call runs in (a different
// device, a context created after a device reset). Only the first call in a
// context loads the module there; later look-ups make no allocation and
// queue no work.
moe_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
  *out = p;
  return MOE_OK;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_permute_static(const moe_config* cfg, const int32_t* topk_idx, const int32_t* counts,
                                         int32_t* offsets, int32_t* sorted_tok, int32_t* slot_pos, const void* x,
                                         void* xp, moe_stream_t stream) {
  if (cfg == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_config& c = *cfg;
  if (c.T < 0 || c.d <= 0 || c.E <= 0 || c.K <= 0 || c.K > 32 || c.E > 512) return MOE_ERR_INVALID_ARG;
  if (c.act != MOE_F32 && c.act != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c.expert != c.act) return MOE_ERR_UNSUPPORTED;  // plain row copies only, no e4m3 tiles
  const size_t row_bytes = (size_t)c.d * (c.act == MOE_F32 ? 4 : 2);
  if (row_bytes % 4 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(offsets)) return MOE_ERR_INVALID_ARG;
  // scratch needed: error word, ranks [T*K], chunk histograms and bases [E * chunks] each
  const size_t TK = (size_t)c.T * c.K;
  const size_t nch = (size_t)moe::permute_chunks(c.T);
  const size_t off_rank = 256;
  const size_t off_hist = off_rank + up256(TK * 4);
  const size_t off_base = off_hist + up256((size_t)c.E * nch * 4);
  const size_t need = off_base + up256((size_t)c.E * nch * 4);
  if (need > MOE_PERMUTE_STATIC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (c.T == 0) {
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1), st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (!aligned16(topk_idx) || !aligned16(counts) || !aligned16(sorted_tok) || !aligned16(slot_pos) ||
      !aligned16(x) || !aligned16(xp))
    return MOE_ERR_INVALID_ARG;
  void* base = nullptr;
  const moe_status s = scratch_address(&base);
  if (s != MOE_OK) return s;
  uint8_t* b = static_cast<uint8_t*>(base);
  int* err = reinterpret_cast<int*>(b);
  int* local_rank = reinterpret_cast<int*>(b + off_rank);
  int* chunk_hist = reinterpret_cast<int*>(b + off_hist);
  int* chunk_base = reinterpret_cast<int*>(b + off_base);
  // Only the error word has to start at zero: ranks, histograms and bases are
  // fully rewritten by every call.
  if (cudaMemsetAsync(err, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  int nsm = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (moe::launch_permute_rank(topk_idx, c.T, c.K, c.E, local_rank, chunk_hist, err, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_permute_scan(counts, chunk_hist, c.T, c.E, chunk_base, offsets, err, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_permute_scatter(topk_idx, local_rank, chunk_base, c.T, c.K, c.E, x, row_bytes, sorted_tok,
                                  slot_pos, xp, nsm, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
