// Epilogues of the tcgen05 bf16 GEMM tiles: one thread per accumulator row
// (TMEM lane), 32 fp32 columns per tcgen05.ld.
#pragma once

#include "gemm_sched.cuh"
#include "gemm_tc.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// Drains the BN accumulator columns of this thread's row at TMEM address
// `tbase` (lane field = the warp's lane quarter) and writes the tile's output.
// bf16 outputs go 32 columns at a time through the warp's staging block `stg`
// (warp_store_rows64); rbase is the warp's first row, nrows how many of its
// 32 rows are stored. Every lane of the warp must call it (tcgen05.ld is
// warp-collective).
template <int BN, Epi EPI>
__device__ __forceinline__ void tile_epilogue(const TcGemmParams& p, const Tile& t, uint32_t tbase, int row,
                                              bool valid, uint8_t* stg, int rbase, int nrows) {
  float v[32];
  if constexpr (EPI == Epi::kRouterSigmoid) {
    float* out = reinterpret_cast<float*>(p.out1);
    const int E = p.n_valid;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      ptx::tmem_ld32(tbase + c * 32, v);
      if (valid) {
        float* dst = out + (size_t)row * E + c * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 1.0f / (1.0f + expf(-v[j]));
        if (c * 32 + 32 <= E && (E % 4) == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4*>(dst)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j < E) dst[j] = v[j];
        }
      }
    }
  } else if constexpr (EPI == Epi::kSwiGLU) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(t.seg ? p.out1 : p.out0);
    const int ldo = t.seg ? p.ldo1 : p.ldo0;
    uint8_t* base = reinterpret_cast<uint8_t*>(out + (size_t)rbase * ldo + t.n * 128);
    float u[32];
    uint4 w[4];
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int gcol = (c >> 1) * 128 + (c & 1) * 32;
      ptx::tmem_ld32(tbase + gcol, v);
      ptx::tmem_ld32(tbase + gcol + 64, u);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = silu(v[j]) * u[j];
      pack_bf16x32(v, w);
      warp_store_rows64(stg, threadIdx.x & 31, w, base + c * 64, (size_t)ldo * 2, nrows);
    }
  } else if constexpr (EPI == Epi::kStore) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out0);
    uint8_t* base = reinterpret_cast<uint8_t*>(out + (size_t)rbase * p.ldo0 + t.n * BN);
    uint4 w[4];
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      ptx::tmem_ld32(tbase + c * 32, v);
      pack_bf16x32(v, w);
      warp_store_rows64(stg, threadIdx.x & 31, w, base + c * 64, (size_t)p.ldo0 * 2, nrows);
    }
  } else {  // kCombine: shared-expert down projection + the routed sum
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out1);
    uint8_t* base = reinterpret_cast<uint8_t*>(out + (size_t)rbase * p.ldo1 + t.n * BN);
    uint4 w[4];
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      ptx::tmem_ld32(tbase + c * 32, v);
      if (valid) add_bf16x32(v, p.radd + (size_t)row * p.ldo1 + t.n * BN + c * 32, 1.0f);
      pack_bf16x32(v, w);
      warp_store_rows64(stg, threadIdx.x & 31, w, base + c * 64, (size_t)p.ldo1 * 2, nrows);
    }
  }
}

}  // namespace
}  // namespace moe
