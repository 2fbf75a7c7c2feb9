/*
 * moe_oracle.h - plain, slow CPU C++ oracle of the DeepSeekMoE layer forward.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU legs load libmoe_oracle.so; the CUDA library never links, includes or
 * calls it, and it shares no code with the CUDA path. It is written as the
 * definition of each step, in loops a reader can check against the pages:
 * double accumulation, no blocking, no fast-math (built with g++ -O2
 * -ffp-contract=off). Worker threads only split independent rows, so every
 * result is the same for any thread count.
 *
 * Sources (tags used in the .cpp):
 *   [digest-2.2]  "DeepSeek-V3技术报告" digest, mpbf.cn/news/71467, section 2.2
 *                 "DeepSeekMoE 与无辅助损失": shared + fine-grained routed
 *                 experts; sigmoid affinities normalised over the K chosen
 *                 experts; top-K on affinity + bias with the gates from the
 *                 raw affinities; the per-step +/- gamma bias update; each
 *                 token uses at most M nodes, chosen by summed affinities; no
 *                 token is dropped; a sequence-level balance loss with a tiny
 *                 weight.
 *   [digest-3.1]  same page, section 3.1 "FP8 混合精度": FP8 GEMM inputs with
 *                 one scale per small tile, higher-precision accumulation.
 *   [resmic-moe]  "DeepSeek-V3架构深度解析", blog.resmic.cn/post/249.html,
 *                 "核心架构二": output = shared-expert sum + gate-weighted
 *                 routed sum; the router is a linear map.
 *
 * Readings where the pages are silent (the same ones the NumPy oracle and the
 * CUDA library take): group score = sum of the group_topk largest biased
 * affinities of the group, added largest first in fp32; ties go to the lower
 * group index, then the lower expert index; the K outputs of a token are
 * ordered by (biased affinity desc, index asc); expert FFN = SwiGLU without
 * biases, W2 (silu(W1 v) * (W3 v)), with w13 holding W1 rows above W3 rows;
 * no residual; the permutation is expert-major, token-ascending; the bias
 * update compares counts_e * E with T * K in integers and adds in fp32; FP8
 * scale = amax / 448 (fp32 division, 1 for an all-zero tile) or, in the
 * power-of-two mode, the smallest 2^e >= amax / 448 with e in [-127, 127];
 * code = e4m3(v / scale), round to nearest even, saturating at 448.
 *
 * Layout: every matrix is dense row-major. threads <= 0 means
 * std::thread::hardware_concurrency().
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Threads that threads <= 0 stands for. */
int mo_hardware_threads(void);

/* s[t, e] = fp32(1 / (1 + exp(-u))), u = fp32(sum_i x[t, i] w_router[e, i])
 * with the sum in double; x [T, d], w_router [E, d], s [T, E]. */
void mo_router_scores(const float* x, int64_t T, int d, const float* w_router, int E, int threads, float* s);

/* Group-limited top-K of every token on s' = s + bias (fp32 add); gates from
 * the raw s. idx, gate [T, K]. */
void mo_select_experts(const float* s, const float* bias, int64_t T, int E, int G, int K, int M, int group_topk,
                       int threads, int32_t* idx, float* gate);

/* Group scores gs [T, G] of s' = s + bias (the first selection step alone). */
void mo_group_scores(const float* s, const float* bias, int64_t T, int E, int G, int group_topk, float* gs);

/* counts[e] = number of (token, slot) pairs with idx == e; counts [E]. */
void mo_expert_counts(const int32_t* idx, int64_t T, int K, int E, int32_t* counts);

/* offsets [E + 1]: exclusive prefix sum of counts. */
void mo_exclusive_offsets(const int32_t* counts, int E, int32_t* offsets);

/* Expert-major, token-ascending positions: sorted_tok [T*K], slot_pos [T, K]. */
void mo_permutation(const int32_t* idx, int64_t T, int K, int E, int32_t* sorted_tok, int32_t* slot_pos);

/* One bias step in place on bias [E] [digest-2.2]. */
void mo_bias_update(const int32_t* counts, int E, int64_t T, int K, float gamma, float* bias);

/* fp32(max_e counts_e * E / (T * K)). */
float mo_load_max_over_mean(const int32_t* counts, int E, int64_t T, int K);

/* Repeated route -> count -> bias update on fixed scores s [T, E]:
 * biases [steps, E] (after each step), idx [steps, T, K], loads [steps]. */
void mo_bias_balancing_loop(const float* s, const float* bias0, int64_t T, int E, int G, int K, int M,
                            int group_topk, int steps, float gamma, int threads, float* biases, int32_t* idx,
                            float* loads);

/* One expert on the rows v [n, d]: y = W2 (silu(W1 v) * (W3 v)), double.
 * w13 [2I, d], w2 [d, I], y [n, d]. */
void mo_swiglu_ffn(const float* v, int64_t n, int d, int I, const float* w13, const float* w2, int threads,
                   double* y);

/* acc[rows[i]] += g[i] * FFN(x[rows[i]]) for i < n (g NULL: gate 1), rows
 * distinct. x [*, d], acc [*, d] double. */
void mo_expert_accumulate(const float* x, int d, const int64_t* rows, int64_t n, int I, const float* w13,
                          const float* w2, const float* g, int threads, double* acc);

/* The whole layer on x [T, d]: scores (from the router, or scores_in when
 * not NULL), routing, out [T, d] = sum_s FFN_s(x) + sum_k gate_k FFN_{e_k}(x)
 * in double (no rounding to the output dtype). w13 [E, 2I, d], w2 [E, d, I],
 * ws13 [S, 2I, d], ws2 [S, d, I]. */
void mo_layer_forward(const float* x, int64_t T, int d, int E, int G, int K, int M, int group_topk, int I, int S,
                      const float* w_router, const float* w13, const float* w2, const float* ws13,
                      const float* ws2, const float* bias, const float* scores_in, int threads, float* scores,
                      int32_t* idx, float* gate, double* out);

/* ---- FP8 e4m3 with per-tile scales [digest-3.1] ---- */

/* Nearest e4m3 value of v (OCP E4M3: bias 7, 3 mantissa bits, max 448, no
 * infinities), ties to even, saturating at +/-448. */
double mo_e4m3_value(float v);
/* Its 8-bit code. */
uint8_t mo_e4m3_code(float v);
/* Value of a code (0x7f and 0xff are NaN). */
double mo_e4m3_decode(uint8_t c);
/* Scale of a tile whose largest magnitude is amax (ue8m0: power-of-two rule). */
float mo_tile_scale(float amax, int ue8m0);

/* 1x128 tiles along each row of v [n, k]: q [n, k] (e4m3 values), scales
 * [n, ceil(k/128)]. */
void mo_quantize_rows_1x128(const float* v, int64_t n, int k, int ue8m0, double* q, float* scales);
/* 128x128 blocks of w [n, k]: q [n, k], scales [ceil(n/128), ceil(k/128)]. */
void mo_quantize_blocks_128x128(const float* w, int64_t n, int k, int ue8m0, double* q, float* scales);
/* out [n, m] = sum over 128-wide K blocks b of (qa_b . qw_b) * sa[r, b] * sw[c/128, b]. */
void mo_fp8_gemm(const double* qa, const float* sa, int64_t n, int k, const double* qw, const float* sw, int64_t m,
                 int threads, double* out);

/* mo_expert_accumulate with e4m3 operands: the expert's master weights are
 * block-quantised, x rows quantised 1x128 along d, GEMM1 in FP8, SwiGLU in
 * double with h rounded to fp32 and re-quantised 1x128 along I, GEMM2 in FP8. */
void mo_expert_accumulate_fp8(const float* x, int d, const int64_t* rows, int64_t n, int I, const float* w13,
                              const float* w2, const float* g, int ue8m0, int threads, double* acc);

/* The FP8 layer: bf16-path routing (router in full precision), then the
 * expert GEMMs in e4m3 as above for every token. Arguments as
 * mo_layer_forward. */
void mo_layer_forward_fp8(const float* x, int64_t T, int d, int E, int G, int K, int M, int group_topk, int I,
                          int S, const float* w_router, const float* w13, const float* w2, const float* ws13,
                          const float* ws2, const float* bias, int ue8m0, int threads, float* scores, int32_t* idx,
                          float* gate, double* out);

/* Sequence-wise balance statistic per run of seq_len tokens: loss [n_seq],
 * f [n_seq, E], P [n_seq, E] (double; f and P may be NULL). */
void mo_sequence_balance(const float* s, const int32_t* idx, int64_t T, int E, int K, int seq_len, double alpha,
                         double* loss, double* f, double* P);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ORACLE_H */
