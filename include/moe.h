/*
 * moe.h - C ABI of the DeepSeekMoE layer forward for NVIDIA B300 (sm_103a).
 *
 * What the layer computes (sources are web pages about the DeepSeek-V3
 * technical report; the tag in brackets is used in every comment below):
 *   [digest-2.2]  "DeepSeek-V3技术报告" digest, mpbf.cn/news/71467, section 2.2
 *                 "DeepSeekMoE 与无辅助损失": shared experts plus fine-grained
 *                 routed experts; sigmoid affinities normalised over the K
 *                 selected experts; top-K on affinity + bias with the gates
 *                 taken from the raw affinities; after each step the bias of
 *                 an overloaded expert drops by gamma and that of an
 *                 underloaded one rises by gamma; each token uses at most M
 *                 nodes, chosen by the summed affinities on each node; no
 *                 token is dropped.
 *   [digest-3.1]  same page, section 3.1 "FP8 混合精度": FP8 GEMM inputs with
 *                 per-tile scale factors and higher-precision accumulation.
 *   [digest-3.3]  same page, section 3.3: the all-to-all dispatch / combine
 *                 that the on-device permutation and combine replace.
 *   [resmic-moe]  "DeepSeek-V3架构深度解析", blog.resmic.cn/post/249.html,
 *                 section "核心架构二": output = shared-expert sum + sum of
 *                 gate-weighted routed experts; the router is a linear map.
 *
 * Notation: T tokens, d hidden width, E routed experts in G equal groups,
 * K experts per token from at most M groups, I expert intermediate width,
 * S shared experts. Expert FFN_e(v) = W2_e (silu(W1_e v) * (W3_e v)).
 *
 * Conventions for every call:
 *   - All tensors are dense, row-major, and live in device memory unless a
 *     parameter says "host". Every pointer must be 16-byte aligned.
 *   - The caller owns all memory. The library allocates nothing on the device:
 *     scratch space comes from `ws`, a device buffer of at least
 *     moe_workspace_size() bytes, which must not be shared by two calls that
 *     run at the same time. Its first 256 bytes must be zero before its first
 *     use (they hold the device error word, see below).
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     Argument errors are reported synchronously, before any work is queued.
 *     A launch failure returns MOE_ERR_CUDA.
 *   - Kernels that wait on on-chip barriers give up after about a second,
 *     write an error code into the first word of `ws` and return; the code is
 *     read back with moe_device_error(). Out-of-range expert indices given to
 *     moe_permute are skipped and reported the same way.
 *   - T == 0 is a valid no-op.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* bad pointer, shape or combination */
  MOE_ERR_UNSUPPORTED = 2,  /* valid layer, but a shape the library does not run */
  MOE_ERR_CUDA = 3,         /* a CUDA runtime / driver call failed */
  MOE_ERR_TIMEOUT = 4,      /* a device-side wait ran out (see moe_device_error) */
  MOE_ERR_DEVICE = 5        /* device-side check failed (see moe_device_error) */
} moe_status;

/* MOE_E4M3: e4m3 codes with fp32 scales, scale = amax / 448 per tile.
 * MOE_E4M3_UE8M0: e4m3 codes whose tile scales are powers of two, the
 *   smallest 2^e >= amax / 448 (e in [-127, 127]; 1 for an all-zero tile),
 *   still passed as fp32 values. The GEMMs then scale inside the tensor
 *   core (tcgen05 block scaling with UE8M0 scale bytes). The scale rule is
 *   this library's option beside the pages' fp32 scales [digest-3.1]; only
 *   the exponent bits of each scale are read. */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_E4M3 = 2, MOE_E4M3_UE8M0 = 3 } moe_dtype;

/* How moe_layer_forward combines the routed experts' rows [resmic-moe]:
 * MOE_COMBINE_GATHER: the routed down projection writes each expert row once
 *   (unscaled, in the workspace); a per-token pass sums the K gated rows of
 *   each token in a fixed order and the shared experts' down projection adds
 *   that sum in its epilogue. Deterministic. With bf16 expert GEMMs and
 *   T*K >= 128*E the layer keeps its permuted rows in a padded layout inside
 *   the workspace (each expert's rows start at a multiple of 128, followed by
 *   zero rows up to it) so that the expert GEMMs' last tile of each expert
 *   multiplies zeros; the results are the same bits as with contiguous rows,
 *   and moe_workspace_size accounts for the 127*E extra rows.
 * MOE_COMBINE_SCATTER_ADD: the shared experts' down projection writes an fp32
 *   [T, d] accumulator, the routed down projection's epilogue adds gate * row
 *   into it with fp32 reductions (red.global.add), and one pass rounds it to
 *   the output dtype (fp32 layers accumulate in out itself). The order of
 *   the K fp32 adds per element is not fixed, so outputs may differ in the
 *   last bits from call to call. bf16 and fp32 layers; layers with FP8
 *   expert GEMMs always gather. */
typedef enum { MOE_COMBINE_GATHER = 0, MOE_COMBINE_SCATTER_ADD = 1 } moe_combine_mode;

typedef struct {
  int T, d, E, G, K, M, I, S;
  int group_topk;     /* group score = sum of this many largest biased
                         affinities in the group, added largest first
                         (2 in DeepSeek-V3 shapes; E/G gives the plain sum
                         over the group's experts, the pages' node score) */
  moe_dtype act;      /* x, out, router weights, yp: MOE_F32 or MOE_BF16 */
  moe_dtype expert;   /* expert GEMM operands: == act, or MOE_E4M3 /
                         MOE_E4M3_UE8M0 with act MOE_BF16 (1x128 activation
                         tiles, 128x128 weight blocks, fp32 accumulation
                         [digest-3.1]) */
  moe_combine_mode combine;  /* moe_layer_forward's combine (see above) */
} moe_config;

/* Expert weights. Element type is cfg->expert (router: cfg->act).
 * w13 holds W1 (rows 0..I-1, the gate projection) above W3 (rows I..2I-1,
 * the up projection) for each expert. For MOE_E4M3 and MOE_E4M3_UE8M0 each
 * weight matrix carries one fp32 scale per 128x128 block: w = code * scale. */
typedef struct {
  const void* w_router;      /* [E, d]   act dtype                  */
  const void* w13;           /* [E, 2I, d]                          */
  const void* w2;            /* [E, d, I]                           */
  const void* ws13;          /* [S, 2I, d]  shared experts          */
  const void* ws2;           /* [S, d, I]                           */
  const float* w13_scale;    /* E4M3: [E, 2I/128, d/128], else NULL */
  const float* w2_scale;     /* E4M3: [E, d/128, I/128]             */
  const float* ws13_scale;   /* E4M3: [S, 2I/128, d/128]            */
  const float* ws2_scale;    /* E4M3: [S, d/128, I/128]             */
} moe_weights;

/* Bytes of device workspace that every call below needs for `cfg`
 * (moe_layer_forward needs the most; one buffer of this size serves all).
 * Limits checked here and by every call: E <= 512 with E % G == 0, G <= 32,
 * 1 <= group_topk <= E/G, K <= 32, K <= M * (E/G), M <= G, d % 128 == 0 and
 * I % 128 == 0; for act BF16 also E <= 256. fp32 layers (act MOE_F32) run
 * their GEMMs on the tensor cores with each fp32 operand split into a tf32
 * pair (high part + remainder; hi*hi + hi*lo + lo*hi), the pairs kept in the
 * workspace (x and the weights are split at the start of every call). */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Router and routing [digest-2.2], [resmic-moe].
 *   scores s = sigmoid(x W_r^T) [T, E] fp32, computed from x [T, d] and
 *   w_router [E, d] unless scores_in (a [T, E] fp32 array) is given, in which
 *   case x and w_router are ignored and s = scores_in.
 *   s' = s + bias (fp32). Group score = sum of the group_topk largest s' of
 *   the group; the M best groups are kept (ties: lower group index); the K
 *   largest s' among their experts are chosen (ties: lower expert index) and
 *   written to topk_idx [T, K] int32 in (s' desc, index asc) order.
 *   topk_gate [T, K] fp32 = s_e / (sum of s over the K chosen experts).
 *   counts [E] int32 = number of (token, slot) pairs per expert; it is zeroed
 *   by this call. scores_out (nullable, [T, E] fp32) receives s.
 *   bias [E] fp32 is read only. */
moe_status moe_route(const moe_config* cfg, const void* x, const void* w_router,
                     const float* scores_in, const float* bias, float* scores_out,
                     int32_t* topk_idx, float* topk_gate, int32_t* counts,
                     void* ws, moe_stream_t stream);

/* Expert-major permutation (the on-device stand-in for the all-to-all
 * dispatch [digest-3.3]; every pair is kept, no token is dropped).
 *   counts [E] must be the histogram of topk_idx (as moe_route writes it).
 *   offsets [E+1] = exclusive scan of counts (offsets[E] = T*K).
 *   Position p in [offsets[e], offsets[e+1]) holds the tokens that chose
 *   expert e, in ascending token order: sorted_tok [T*K] gives the token at p,
 *   slot_pos [T, K] gives the position of slot k of token t.
 *   xp [T*K, d] receives the gathered rows x[sorted_tok[p]] in cfg->act, or
 *   for MOE_E4M3 the e4m3 codes of the 1x128 tiles of those rows with their
 *   scales in xp_scale, laid out [d/128, T*K] (tile-major); xp_scale is NULL
 *   otherwise. */
moe_status moe_permute(const moe_config* cfg, const int32_t* topk_idx, const int32_t* counts,
                       int32_t* offsets, int32_t* sorted_tok, int32_t* slot_pos,
                       const void* x, void* xp, float* xp_scale,
                       void* ws, moe_stream_t stream);

/* Routed experts on the permuted rows [digest-2.2]:
 *   yp[p] = FFN_e(xp[p]) for every p in [offsets[e], offsets[e+1]),
 *   yp [T*K, d] in cfg->act, not yet scaled by the gates. offsets is read on
 *   the device, so no host synchronisation is needed after moe_permute. */
moe_status moe_grouped_ffn(const moe_config* cfg, const void* xp, const float* xp_scale,
                           const int32_t* offsets, const moe_weights* w, void* yp,
                           void* ws, moe_stream_t stream);

/* Shared experts and gate-weighted combine [resmic-moe]:
 *   out[t] = sum_s FFN_s(x[t]) + sum_k topk_gate[t,k] * yp[slot_pos[t,k]]
 *   out [T, d] in cfg->act. The routed sum is added in the epilogue of the
 *   shared experts' down projection. x [T, d] in cfg->act. */
moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* slot_pos,
                       const float* topk_gate, const void* x, const moe_weights* w,
                       void* out, void* ws, moe_stream_t stream);

/* Auxiliary-loss-free bias update [digest-2.2], in place on bias [E] fp32:
 *   counts_e * E >  T*K  ->  bias_e -= gamma   (overloaded)
 *   counts_e * E <  T*K  ->  bias_e += gamma   (underloaded)
 *   otherwise unchanged. The comparison is exact (integers); the add is fp32.
 *   max_over_mean (nullable, device, 1 float) = max_e counts_e * E / (T*K). */
moe_status moe_bias_update(const moe_config* cfg, const int32_t* counts, float gamma,
                           float* bias, float* max_over_mean, moe_stream_t stream);

/* The whole layer: route, permute, routed experts, shared experts with the
 * fused combine (cfg->combine chooses how, see moe_combine_mode), and (when
 * gamma != 0) the bias update, queued on `stream`. The shared experts' first
 * GEMM (and, with MOE_COMBINE_SCATTER_ADD, their down projection) runs on an
 * internal side stream (one per host thread and device, created by the first
 * call and kept until the process exits) while `stream` routes and permutes;
 * `stream` waits for it before the combine, so the layer is complete when
 * `stream` is. Make the
 * first call on a device outside stream capture; later calls may be
 * captured into a CUDA graph (the side stream's fork and join become graph
 * edges, and the call makes no allocation or attribute change) and the graph
 * replayed, each replay one step on the buffers given at capture time.
 * out [T, d] in cfg->act; topk_idx, topk_gate, counts as in moe_route;
 * bias [E] fp32 is updated in place after routing when gamma != 0;
 * max_over_mean as in moe_bias_update (nullable). */
moe_status moe_layer_forward(const moe_config* cfg, const void* x, const moe_weights* w,
                             float* bias, float gamma, void* out, int32_t* topk_idx,
                             float* topk_gate, int32_t* counts, float* max_over_mean,
                             void* ws, moe_stream_t stream);

/* 128x128 block quantisation of n_mat bf16 matrices [n_mat, rows, cols] to
 * e4m3 codes q (same shape, 1 byte each) and fp32 scales
 * [n_mat, ceil(rows/128), ceil(cols/128)]: scale = amax / 448 (1 if the block
 * is all zero), code = e4m3(w / scale) rounded to nearest even and saturated
 * to +/-448 [digest-3.1]. Used to prepare MOE_E4M3 expert weights. */
moe_status moe_quantize_weights_e4m3(const void* w, int n_mat, int rows, int cols,
                                     uint8_t* q, float* scale, moe_stream_t stream);

/* The same with power-of-two scales: scale = the smallest 2^e >= amax / 448,
 * e in [-127, 127] (1 if the block is all zero), code = e4m3(w / scale).
 * Used to prepare MOE_E4M3_UE8M0 expert weights. */
moe_status moe_quantize_weights_e4m3_ue8m0(const void* w, int n_mat, int rows, int cols,
                                           uint8_t* q, float* scale, moe_stream_t stream);

/* Sequence-wise balance statistic of a routing [digest-2.2: the sequence-level
 * balance loss kept with a tiny weight; its formula is the DeepSeek-V3
 * report's]. For each run of seq_len consecutive tokens (the last run may be
 * shorter; L = its length):
 *   f_i  = E / (K L) * (number of tokens of the run whose K choices include i)
 *   P_i  = (1 / L) * sum_t s_{i,t} / sum_j s_{j,t}     (raw affinities)
 *   loss = alpha * sum_i f_i P_i
 *   scores:   [T, E] fp32 affinities, device, 16-byte aligned; NULL to use the
 *             ones the last moe_route / moe_layer_forward call on ws left there
 *   topk_idx: [T, K] int32 chosen experts (entries outside [0, E) are not counted)
 *   loss:     [ceil(T/seq_len)] fp32 out; f, p: [ceil(T/seq_len), E] fp32 out
 *             or NULL. Forward only (no gradient); deterministic.
 * MOE_ERR_INVALID_ARG for seq_len <= 0 or bad pointers. */
moe_status moe_seq_balance(const moe_config* cfg, const float* scores, const int32_t* topk_idx, int seq_len,
                           float alpha, float* loss, float* f, float* p, void* ws, moe_stream_t stream);

/* Row moves for expert-parallel dispatch and combine [digest-3.3: tokens are
 * sent to the GPUs that hold their experts and the expert outputs are sent
 * back]. A rank's moe_permute output is already ordered by destination rank
 * (experts are placed in contiguous blocks per rank), and the rows it receives
 * arrive source-major; these two calls reorder them for the rank's grouped
 * expert GEMMs and back:
 *   moe_gather_rows:  dst[i] = src[idx[i]] for i < n (src holds n_src rows);
 *   moe_scatter_rows: dst[idx[i]] = src[i] for i < n (dst holds n_dst rows).
 * Rows are row_bytes long (a multiple of 4), src and dst 16-byte aligned
 * device buffers owned by the caller, idx [n] int32 on the device. An index
 * outside the other buffer's rows is skipped and reported as code 0x203 in
 * the error word of ws (any workspace of moe_workspace_size bytes; read it
 * with moe_device_error). A scatter index that repeats leaves one of the
 * rows written to it, which one unspecified. n == 0 is a no-op. Asynchronous
 * on stream. MOE_ERR_INVALID_ARG for bad pointers or sizes. */
moe_status moe_gather_rows(const void* src, int n_src, const int32_t* idx, int n, size_t row_bytes, void* dst,
                           void* ws, moe_stream_t stream);
moe_status moe_scatter_rows(const void* src, const int32_t* idx, int n, size_t row_bytes, void* dst, int n_dst,
                            void* ws, moe_stream_t stream);

/* CUDA-graph replay of moe_layer_forward (on by default; the environment
 * variable MOE_LAYER_GRAPHS=0 starts the process with it off). When on, the
 * second call with the same configuration, pointers, gamma and stage-event
 * setting (moe_set_stage_events on or off) on the same CUDA context is
 * captured into a graph, and that call and every later one with the same
 * arguments replay it with one cudaGraphLaunch on the caller's stream: the
 * same kernels with the same arguments, so the same results, without the
 * per-kernel launch gaps. The events given to moe_set_stage_events are
 * re-targeted on each replay. Calls on a stream that is itself being captured
 * run the kernels directly (they become part of the caller's graph). Up to 16
 * argument sets are kept per process, the least recently used one replaced
 * by a new one. A graph holds the pointers it was captured with: a buffer
 * freed and reallocated at the same address with the same configuration is
 * used as the new buffer, as with any cached launch.
 * enable: 1 on, 0 off (the kept graphs stay, unused). MOE_ERR_INVALID_ARG
 * for other values. */
moe_status moe_set_layer_graphs(int enable);
/* Number of argument sets that moe_layer_forward currently replays from a
 * graph (written to *n). */
moe_status moe_layer_graphs_kept(int* n);

/* Bytes of the fixed device array that moe_permute_static uses as scratch. */
#define MOE_PERMUTE_STATIC_SCRATCH_BYTES (4u << 20)

/* moe_permute without a workspace, for callers that cannot allocate device
 * memory: code that is handed only its input and output buffers by a host
 * framework with no scratch hook (a plugin inside another engine, say), or
 * that runs where device allocation after start-up is not allowed (a fixed
 * memory budget set once at start). There is no counterpart on the pages; it
 * is a packaging variant of moe_permute for such callers.
 *   Same inputs and outputs as moe_permute for act == expert (row copies; no
 *   e4m3 tiles). Scratch comes from one static device array of
 *   MOE_PERMUTE_STATIC_SCRATCH_BYTES (4 MiB) that every GPU which loads the
 *   library keeps until the process exits. A call needs
 *   256 + 4*T*K + 8*E*ceil(T/32) bytes of it (each part rounded up to 256);
 *   larger calls return MOE_ERR_UNSUPPORTED before any work is queued
 *   (T = 16384, K = 8, E = 256 needs 1.5 MiB; T = 32768 needs 3 MiB).
 *   The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *   library routine.
 *   Every call asks cudaGetSymbolAddress for the array's address in the
 *   current device's context, so the address always belongs to that context
 *   (also after a device reset). The first call in a context loads the
 *   library's device code there; make that first call before any stream
 *   capture.
 *   All calls on a device share the one array and leave their contents in it;
 *   each call clears the part that must start at zero. Calls whose work
 *   overlaps on the GPU (other streams, other host threads) race on the array
 *   and must be serialised by the caller. Out-of-range expert indices are
 *   skipped, but not reported (moe_device_error does not see this array). */
moe_status moe_permute_static(const moe_config* cfg, const int32_t* topk_idx, const int32_t* counts,
                              int32_t* offsets, int32_t* sorted_tok, int32_t* slot_pos,
                              const void* x, void* xp, moe_stream_t stream);

/* Profiling hook. After this call, every moe_layer_forward made from the
 * calling thread records events[i] (cudaEvent_t handles owned by the caller)
 * on its stream at stage boundary i: 0 before the router, 1 after the router
 * GEMM, 2 after the top-K selection, 3 after the permutation, 4 after the
 * routed experts' GEMM1 (SwiGLU), 5 after the routed down projection, 6 after
 * the combine (gather: the routed sum and the shared down projection that
 * adds it; scatter-add: the rounding of the accumulator), 7 after the bias
 * update. The side stream's work starts at mark 1 and is joined between
 * marks 5 and 6 (gather) or 4 and 5 (scatter-add), so the stages in between
 * share the GPU with it. count must be 0 (hook off) or >= 8. */
moe_status moe_set_stage_events(void* const* events, int count);

/* Self-test of the device-side wait bound: queues one small kernel that waits
 * on an on-chip barrier nothing will release. The wait gives up after about a
 * second, records MOE_ERR_TIMEOUT's device code (0x105) in the error word of
 * `ws` and the kernel exits; read it with moe_device_error. */
moe_status moe_selftest_timeout(void* ws, moe_stream_t stream);

/* Synchronises `stream`, then reads and clears the device error word in `ws`.
 * *code receives 0 when no device-side check has fired since the last call;
 * the return value is MOE_ERR_TIMEOUT / MOE_ERR_DEVICE when one has. */
moe_status moe_device_error(void* ws, moe_stream_t stream, int* code);

/* Static description of a status code. */
const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
