// FP8 (e4m3) grouped GEMMs on tcgen05 with 1x128 / 128x128 scales: fp32
// promotion of every 128-wide K block (gemm_fp8.cu), or tensor-core block
// scaling for power-of-two scales (gemm_mx.cu).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {

enum class Fp8Epi : int {
  kSwiGLU = 0,   // h = silu(gate) * up, written as e4m3 1x128 tiles + scales
  kStore = 1,    // bf16 out = acc
  kCombine = 2,  // bf16 out = acc + radd
};

struct Fp8GemmParams {
  int groups0;
  const int* offsets0;
  int rows_total0;          // rows of the segment-0 A matrix (scale layout stride)
  int rows1;
  int n_tiles0, n_tiles1;
  int k_blocks0, k_blocks1;  // K / 128 per segment
  int I;                    // expert intermediate width
  int N;                    // down projection: output width d
  const float* a_scale0;    // [K/128, rows_total0]
  const float* a_scale1;    // [K/128, rows1]
  const float* b_scale0;    // weight block scales of segment 0
  const float* b_scale1;    // ... of segment 1 (shared experts)
  void* out0;
  void* out1;
  int ldo0, ldo1;
  float* out_scale0;        // kSwiGLU: [I/128, rows_total0]
  float* out_scale1;        // kSwiGLU: [S*I/128, rows1]
  const __nv_bfloat16* radd;  // kCombine: [rows1, ldo1]
  int* err;
};

struct Fp8GemmLaunch {
  Fp8Epi epi;
  CUtensorMap a0, b0, a1, b1;
  Fp8GemmParams p;
  int grid;
  cudaStream_t stream;
};

cudaError_t launch_fp8_gemm(const Fp8GemmLaunch& L);

// Same operands and epilogues with power-of-two scales, scaled inside the
// tensor core (gemm_mx.cu).
cudaError_t launch_mx_gemm(const Fp8GemmLaunch& L);

}  // namespace moe
