// Shared definitions of the CUDA side of the MoE layer library.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

namespace moe {

// Device error word codes (first int of the workspace).
enum DevErr : int {
  kDevOk = 0,
  kDevTimeoutProducer = 0x101,   // TMA producer gave up waiting for a free stage
  kDevTimeoutMma = 0x102,        // MMA issuer gave up waiting for data / TMEM
  kDevTimeoutEpilogue = 0x103,   // epilogue gave up waiting for an accumulator
  kDevTimeoutDrain = 0x104,      // exit-time wait for in-flight copies ran out
  kDevTimeoutSelfTest = 0x105,   // moe_selftest_timeout: the wait ran out as intended
  kDevBadExpertIndex = 0x201,    // topk_idx entry outside [0, E)
  kDevCountMismatch = 0x202,     // counts[] is not the histogram of topk_idx
  kDevBadRowIndex = 0x203,       // moe_gather_rows / moe_scatter_rows: row index out of range
};

// A device-side wait that sees no progress for this long gives up.
constexpr unsigned long long kWaitTimeoutNs = 1000000000ull;  // 1 s
constexpr long long kWaitTimeoutCycles = 8000000000ll;          // 4 s at 2 GHz: backstop only

struct __align__(16) bf16x8 {
  __nv_bfloat162 v[4];
};

__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ int read_error(const int* err) {
  return err ? *reinterpret_cast<const volatile int*>(err) : 0;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// silu with the hardware exp2 and reciprocal approximations (a few fp32 ulp,
// far below the bf16 / e4m3 rounding of the SwiGLU output h).
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Scale of one e4m3 tile whose largest magnitude is amax; 1 for an all-zero
// tile. The fp32 rule is amax / 448. The UE8M0 rule is the smallest power of
// two 2^e >= amax / 448 with e clamped to [-127, 127] (the exponents a UE8M0
// byte holds), read off the bits of amax: amax = 1.f * 2^(x - 127) and
// 448 = 1.75 * 2^8, so 2^(x - 135) is the answer unless 1.f > 1.75, when it
// is twice that. 2^-127 is returned as the fp32 subnormal 0x00400000.
__device__ __forceinline__ float e4m3_tile_scale(float amax, bool ue8m0) {
  if (!(amax > 0.0f)) return 1.0f;
  if (!ue8m0) return __fdiv_rn(amax, 448.0f);
  const uint32_t b = __float_as_uint(amax);
  const int x = (int)(b >> 23);
  int e = x == 0 ? -127 : x - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  e = max(-127, min(127, e));
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// UE8M0 byte (biased exponent, 2^-127 -> 0) of a positive power-of-two scale.
// The mantissa bits of any other value are ignored.
__device__ __forceinline__ uint32_t ue8m0_byte(float s) { return (__float_as_uint(s) >> 23) & 0xFFu; }

// Raises the dynamic shared-memory limit of `kern` on the current device the
// first time it is asked there (`done` is one array per kernel
// instantiation), so that later launches, including launches issued while a
// stream is being captured into a CUDA graph, make no attribute call.
template <typename F>
inline cudaError_t set_smem_once(F kern, int bytes, int (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
  return e;
}

// Selection key of a biased affinity v of expert e: the order-preserving bits
// of v above the complement of e, so that the larger key is the larger value
// and, among equal values, the lower expert index. -0 and +0 share a key.
__device__ __forceinline__ uint64_t score_key(float v, int e) {
  if (v == 0.0f) v = 0.0f;
  uint32_t b = __float_as_uint(v);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)b << 32) | (uint32_t)(~(uint32_t)e);
}

// High part of x for the three-product tf32 GEMMs: x rounded to the nearest
// value with 10 mantissa bits (which tf32 holds exactly; ties away from
// zero). x - tf32_hi(x) is exact in fp32 and at most 2^-11 |x|.
__device__ __forceinline__ float tf32_hi(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// e4m3 code of v (round to nearest even, saturating to +/-448).
__device__ __forceinline__ uint8_t f32_to_e4m3(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

}  // namespace moe
