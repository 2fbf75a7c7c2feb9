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
// With SPLIT (fp32 operands as tf32 pairs) the outputs are fp32: the SwiGLU
// rows are written as tf32 pairs ([rows, 2, ldo]: high parts, then
// remainders) for the down projection that reads them, and the combine adds
// an fp32 routed sum.
template <int BN, Epi EPI, bool SPLIT = false>
__device__ __forceinline__ void tile_epilogue(const TcGemmParams& p, const Tile& t, uint32_t tbase, int row,
                                              bool valid, uint8_t* stg, int rbase, int nrows) {
  float v[32];
  if constexpr (EPI == Epi::kRouterSigmoid) {
    // tile n covers experts n*BN .. n*BN + BN - 1
    float* out = reinterpret_cast<float*>(p.out1);
    const int E = p.n_valid;
    const int e0 = t.n * BN;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      ptx::tmem_ld32(tbase + c * 32, v);
      if (valid) {
        float* dst = out + (size_t)row * E + e0 + c * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 1.0f / (1.0f + expf(-v[j]));
        if (e0 + c * 32 + 32 <= E && (E % 4) == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4*>(dst)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (e0 + c * 32 + j < E) dst[j] = v[j];
        }
      }
    }
  } else if constexpr (EPI == Epi::kSwiGLU && SPLIT) {
    // h = silu(gate) * up in fp32, written as tf32 pairs [rows, 2, ldo]
    float* out = reinterpret_cast<float*>(t.seg ? p.out1 : p.out0);
    const int ldo = t.seg ? p.ldo1 : p.ldo0;
    float* hi_base = out + (size_t)rbase * 2 * ldo + t.n * 128;
    float u[32];
    uint4 wh[4], wl[4];
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int gcol = (c >> 1) * 128 + (c & 1) * 32;
      ptx::tmem_ld32(tbase + gcol, v);
      ptx::tmem_ld32(tbase + gcol + 64, u);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = silu(v[j]) * u[j];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float hv[4], lv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            hv[i] = tf32_hi(v[16 * h + 4 * q + i]);
            lv[i] = v[16 * h + 4 * q + i] - hv[i];
          }
          wh[q] = make_uint4(__float_as_uint(hv[0]), __float_as_uint(hv[1]), __float_as_uint(hv[2]),
                             __float_as_uint(hv[3]));
          wl[q] = make_uint4(__float_as_uint(lv[0]), __float_as_uint(lv[1]), __float_as_uint(lv[2]),
                             __float_as_uint(lv[3]));
        }
        float* col = hi_base + c * 32 + 16 * h;
        warp_store_rows64(stg, threadIdx.x & 31, wh, reinterpret_cast<uint8_t*>(col), (size_t)ldo * 8, nrows);
        warp_store_rows64(stg, threadIdx.x & 31, wl, reinterpret_cast<uint8_t*>(col + ldo), (size_t)ldo * 8, nrows);
      }
    }
  } else if constexpr (EPI == Epi::kCombine && SPLIT) {
    // fp32 shared-expert down projection + the fp32 routed sum
    float* out = reinterpret_cast<float*>(p.out1);
    float* base = out + (size_t)rbase * p.ldo1 + t.n * BN;
    uint4 w[4];
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      ptx::tmem_ld32(tbase + c * 32, v);
      if (valid) {
        const float4* r4 = reinterpret_cast<const float4*>(p.radd_f32 + (size_t)row * p.ldo1 + t.n * BN + c * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 a = __ldg(r4 + q);
          v[4 * q] += a.x;
          v[4 * q + 1] += a.y;
          v[4 * q + 2] += a.z;
          v[4 * q + 3] += a.w;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[q] = make_uint4(__float_as_uint(v[16 * h + 4 * q]), __float_as_uint(v[16 * h + 4 * q + 1]),
                            __float_as_uint(v[16 * h + 4 * q + 2]), __float_as_uint(v[16 * h + 4 * q + 3]));
        warp_store_rows64(stg, threadIdx.x & 31, w, reinterpret_cast<uint8_t*>(base + c * 32 + 16 * h),
                          (size_t)p.ldo1 * 4, nrows);
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
      for (int j = 0; j < 32; ++j) v[j] = silu_fast(v[j]) * u[j];
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
  } else if constexpr (EPI == Epi::kStoreF32) {
    // fp32 rows, 16 columns (64 bytes) per staged store
    float* out = reinterpret_cast<float*>(t.seg ? p.out1 : p.out0);
    const int ldo = t.seg ? p.ldo1 : p.ldo0;
    uint8_t* base = reinterpret_cast<uint8_t*>(out + (size_t)rbase * ldo + t.n * BN);
    uint4 w[4];
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      ptx::tmem_ld32(tbase + c * 32, v);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[q] = make_uint4(__float_as_uint(v[16 * h + 4 * q]), __float_as_uint(v[16 * h + 4 * q + 1]),
                            __float_as_uint(v[16 * h + 4 * q + 2]), __float_as_uint(v[16 * h + 4 * q + 3]));
        warp_store_rows64(stg, threadIdx.x & 31, w, base + c * 128 + h * 64, (size_t)ldo * 4, nrows);
      }
    }
  } else if constexpr (EPI == Epi::kScatterAdd) {
    // routed down projection with the combine: each row p belongs to token
    // sorted_tok[p] with gate gate_p[p]; gate * row is added to that token's
    // fp32 output row
    float* acc = reinterpret_cast<float*>(p.out0) + (size_t)t.n * BN;
    const int tok = valid ? __ldg(p.sorted_tok + row) : 0;
    const float g = valid ? __ldg(p.gate_p + row) : 0.0f;
    uint4 w[4];
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      ptx::tmem_ld32(tbase + c * 32, v);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[q] = make_uint4(__float_as_uint(g * v[16 * h + 4 * q]), __float_as_uint(g * v[16 * h + 4 * q + 1]),
                            __float_as_uint(g * v[16 * h + 4 * q + 2]), __float_as_uint(g * v[16 * h + 4 * q + 3]));
        warp_red_rows64(stg, threadIdx.x & 31, w, acc + c * 32 + h * 16, tok, (size_t)p.ldo0, nrows);
      }
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
