// Host-side launchers of the library's kernels (one translation unit each).
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>

#include "common.cuh"

namespace moe {

// ---- routing (route.cu)
cudaError_t launch_route_select(const float* scores, const float* bias, int T, int E, int G, int K, int M, int gk,
                                int* topk_idx, float* topk_gate, int* counts, int num_sms, cudaStream_t st);
cudaError_t launch_router_f32(const float* x, const float* wr, int T, int d, int E, float* scores, cudaStream_t st);
cudaError_t launch_seq_balance(const float* scores, const int* topk_idx, int T, int E, int K, int seq_len,
                               float alpha, float* loss, float* f, float* p, cudaStream_t st);

// ---- permutation (permute.cu)
int permute_chunks(int T);
cudaError_t launch_permute_rank(const int* topk_idx, int T, int K, int E, int* local_rank, int* chunk_hist, int* err,
                                cudaStream_t st);
cudaError_t launch_permute_scan(const int* counts, const int* chunk_hist, int T, int E, int* chunk_base, int* offsets,
                                int* err, cudaStream_t st);
cudaError_t launch_permute_scatter(const int* topk_idx, const int* local_rank, const int* chunk_base, int T, int K,
                                   int E, const void* x, size_t row_bytes, int* sorted_tok, int* slot_pos, void* xp,
                                   int num_sms, cudaStream_t st);
cudaError_t launch_permute_scatter_e4m3(const int* topk_idx, const int* local_rank, const int* chunk_base, int T,
                                        int K, int E, const __nv_bfloat16* x, int d, int* sorted_tok, int* slot_pos,
                                        uint8_t* xp, float* xp_scale, uint8_t* xq, float* xq_scale, float* tok_scale,
                                        bool ue8m0, int num_sms, cudaStream_t st);

// ---- bias update and quantisers (bias_quant.cu)
cudaError_t launch_bias_update(const int* counts, int E, long long TK, float gamma, float* bias,
                               float* max_over_mean, cudaStream_t st);
cudaError_t launch_quantize_blocks(const __nv_bfloat16* w, int n_mat, int rows, int cols, uint8_t* q, float* scale,
                                   bool ue8m0, cudaStream_t st);
cudaError_t launch_quantize_rows(const __nv_bfloat16* x, int rows, int d, uint8_t* q, float* scale, bool ue8m0,
                                 int num_sms, cudaStream_t st);

// ---- fp32 expert GEMMs (gemm_simt.cu)
enum SimtMode : int { kSimtSwiGLU = 0, kSimtStore = 1, kSimtCombine = 2 };

struct SimtParams {
  int mode;
  const float* A;
  int lda;
  const float* B;       // W13 [groups, 2I, d] (SwiGLU) or W2 [groups, d, I]
  int groups;           // > 0: routed groups with device offsets
  const int* offsets;
  int rows;             // groups == 0: one group of this many rows
  int shared;           // 1: the groups are S shared experts concatenated along I
  int N;                // output columns
  int Kdim;             // contraction length
  int I;
  float* out;
  int ldo;
  const int* slot_pos;  // kSimtCombine
  const float* gate;
  const float* yp;
  int topk;
};

cudaError_t launch_simt_gemm(const SimtParams& p, int max_mtiles, cudaStream_t st);
int simt_max_mtiles(int rows_total, int groups);
cudaError_t launch_routed_sum_bf16(const void* yp, const int* slot_pos, const float* gate, int T, int d, int topk,
                                   void* r, int num_sms, cudaStream_t st);
cudaError_t launch_gather_combine(const void* yp, const int* slot_pos, const float* gate, int T, int d, int topk,
                                  bool bf16, void* out, int num_sms, cudaStream_t st);

}  // namespace moe
