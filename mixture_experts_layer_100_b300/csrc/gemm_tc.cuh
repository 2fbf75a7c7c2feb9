// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05) for
// sm_103a, bf16 operands (or fp32 operands as tf32 pairs), fp32 accumulation
// in tensor memory.
//
// C[row, n] = sum_k A[row, k] * B_g[n, k] for every row of group g. Both
// operands are K-major and are moved global -> shared by TMA with 128-byte
// swizzle. Work is split into 128 x BN output tiles; one CTA per SM walks the
// tile list with a static stride. Warp roles inside a CTA (192 threads):
//   warp 0      TMA producer (one lane): fills a STAGES-deep ring of A/B tiles
//   warp 1      MMA issuer (one lane): tcgen05.mma into one of two TMEM
//               accumulators, tcgen05.commit frees ring slots / signals tiles
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, fused math,
//               stores to global memory
// Two accumulators (2 x BN TMEM columns) let the epilogue of tile i overlap
// the main loop of tile i+1.
//
// A launch covers up to two segments that share the epilogue:
//   segment 0: `groups0` groups with device-side row offsets (routed experts
//              on the expert-major permuted rows; the group sizes are read on
//              the device, so no host synchronisation is needed);
//   segment 1: one group of `rows1` rows (shared experts or the router).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {

enum class Epi : int {
  kRouterSigmoid = 0,  // out fp32 [rows, n_valid] = sigmoid(acc)
  kSwiGLU = 1,         // out bf16 [rows, ldo] = silu(gate) * up  (128 cols per tile)
  kStore = 2,          // out bf16 [rows, ldo] = acc
  kCombine = 3,        // out bf16 [T, ldo] = acc + radd (the gate-weighted routed sum)
  kStoreF32 = 4,       // out fp32 [rows, ldo] = acc
  kScatterAdd = 5,     // out fp32 [T, ldo]: out[sorted_tok[row]] += gate_p[row] * acc (reductions)
};

struct TcGemmParams {
  int groups0;          // segment 0 groups (0: no segment 0)
  const int* offsets0;  // [groups0 + 1] device row offsets of segment 0
  // [groups0] or NULL: rows of each group that are written (the padded
  // layout's groups end with zero rows that are multiplied but not stored)
  const int* counts0;
  int rows1;            // rows of segment 1 (0: no segment 1)
  int n_tiles0, n_tiles1;
  int k_blocks0, k_blocks1;  // K / 64 per segment
  int I;                // expert intermediate width (B row / K addressing)
  void* out0;
  void* out1;
  int ldo0, ldo1;       // output row strides (elements)
  int n_valid;          // router: number of experts (output columns)
  // kCombine: per-token routed sum r[t] = sum_k gate[t,k] * yp[slot_pos[t,k]],
  // [T, ldo1] bf16, added to the shared experts' output in the epilogue
  const __nv_bfloat16* radd;
  const float* radd_f32;  // kCombine with fp32 (tf32-pair) operands: fp32 [T, ldo1]
  // kScatterAdd: token of each permuted row and its gate (segment 0 rows)
  const int* sorted_tok;
  const float* gate_p;
  int* err;             // device error word
};

struct TcGemmLaunch {
  Epi epi;
  int bn;
  int mh = 1;  // 128-row halves per tile (expert GEMMs: 1 or 2)
  // fp32 operands as tf32 pairs: every operand row holds its tf32 high part
  // and its remainder ([.., 2, K]); the product is taken as hi*hi + hi*lo +
  // lo*hi with kind::tf32 MMAs
  bool split = false;
  CUtensorMap a0, b0, a1, b1;
  TcGemmParams p;
  int grid;
  cudaStream_t stream;
};

// Queues one launch; returns the launch status.
cudaError_t launch_tc_gemm(const TcGemmLaunch& L);

}  // namespace moe
