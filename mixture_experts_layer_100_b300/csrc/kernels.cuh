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
cudaError_t launch_seq_balance(const float* scores, const int* topk_idx, int T, int E, int K, int seq_len,
                               float alpha, float* loss, float* f, float* p, cudaStream_t st);

// ---- permutation (permute.cu)
int permute_chunks(int T);
cudaError_t launch_permute_rank(const int* topk_idx, int T, int K, int E, int* local_rank, int* chunk_hist, int* err,
                                cudaStream_t st);
// pad > 1: every expert's block of rows starts at a multiple of pad (its
// rows followed by up to pad - 1 unused rows), which the scatter fills with
// zeros (given offsets and counts).
cudaError_t launch_permute_scan(const int* counts, const int* chunk_hist, int T, int E, int* chunk_base, int* offsets,
                                int* err, cudaStream_t st, int pad = 1);
cudaError_t launch_permute_scatter(const int* topk_idx, const int* local_rank, const int* chunk_base, int T, int K,
                                   int E, const void* x, size_t row_bytes, int* sorted_tok, int* slot_pos, void* xp,
                                   int num_sms, cudaStream_t st, const float* gate_in = nullptr,
                                   float* gate_p = nullptr, int pad = 1, const int* offsets = nullptr,
                                   const int* counts = nullptr);
cudaError_t launch_permute_scatter_e4m3(const int* topk_idx, const int* local_rank, const int* chunk_base, int T,
                                        int K, int E, const __nv_bfloat16* x, int d, int* sorted_tok, int* slot_pos,
                                        uint8_t* xp, float* xp_scale, uint8_t* xq, float* xq_scale, float* tok_scale,
                                        bool ue8m0, int num_sms, cudaStream_t st, const float* gate_in = nullptr,
                                        float* gate_p = nullptr);

// Rows moved by an index list (row_bytes a multiple of 4): gather dst[i] =
// src[idx[i]] (n_other = rows of src) or scatter dst[idx[i]] = src[i]
// (n_other = rows of dst); out-of-range indices are skipped and reported.
cudaError_t launch_move_rows(const void* src, const int* idx, int n, int n_other, size_t row_bytes, void* dst,
                             bool gather, int* err, int num_sms, cudaStream_t st);

// ---- bias update and quantisers (bias_quant.cu)
cudaError_t launch_bias_update(const int* counts, int E, long long TK, float gamma, float* bias,
                               float* max_over_mean, cudaStream_t st);
cudaError_t launch_quantize_blocks(const __nv_bfloat16* w, int n_mat, int rows, int cols, uint8_t* q, float* scale,
                                   bool ue8m0, cudaStream_t st);
// fp32 rows [rows, cols] -> [rows, 2 cols]: each row's tf32 high part, then
// the remainder (cols % 4 == 0).
cudaError_t launch_split_tf32(const float* src, long long rows, int cols, float* dst, int num_sms, cudaStream_t st);
cudaError_t launch_quantize_rows(const __nv_bfloat16* x, int rows, int d, uint8_t* q, float* scale, bool ue8m0,
                                 int num_sms, cudaStream_t st);

// ---- combine passes (combine.cu)
cudaError_t launch_routed_sum_bf16(const void* yp, const int* slot_pos, const float* gate, int T, int d, int topk,
                                   void* r, int num_sms, cudaStream_t st);
// out [n] bf16 = round(acc [n] fp32), n a multiple of 8 (the scatter-add
// combine's last pass).
cudaError_t launch_acc_to_bf16(const float* acc, size_t n, void* out, int num_sms, cudaStream_t st);
cudaError_t launch_gather_combine(const void* yp, const int* slot_pos, const float* gate, int T, int d, int topk,
                                  bool bf16, void* out, int num_sms, cudaStream_t st);

}  // namespace moe
