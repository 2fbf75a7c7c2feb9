"""CPU oracle for the DeepSeekMoE layer forward.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import or run this module. The product path
(the CUDA library and its Python binding) never does, and shares no code
with it: this file is a plain, slow, float64 restatement of what the layer
computes, written so that each step can be checked against the pages by eye.

Sources (cited below by the tag in brackets):
  [digest-2.2]  "DeepSeek-V3技术报告" digest, mpbf.cn/news/71467,
                section 2.2 "DeepSeekMoE 与无辅助损失" (shared + fine-grained
                routed experts, sigmoid affinities normalised over the selected
                experts, bias used only for the top-K decision, per-step
                +/- gamma bias update, node-limited routing by summed
                affinities, no token dropping).
  [digest-3.1]  same page, section 3.1 "FP8 混合精度" (FP8 GEMM inputs with
                per-tile scale factors, higher-precision accumulation).
  [digest-3.3]  same page, section 3.3 (at most 4 nodes per token; 8 routed
                experts per token).
  [resmic-moe]  "DeepSeek-V3架构深度解析", blog.resmic.cn/post/249.html,
                section "核心架构二: DeepSeekMoE" (the layer output is the
                shared-expert sum plus the gate-weighted routed sum; the
                router is a linear map of the hidden state).
  [p2hp-2]      "Deepseek-v3技术报告简报", p2hp.com/show/183.html, section 2
                (256 routed + 1 shared expert, top-8, width 7168).

Readings where the pages are silent (each is listed in the design notes):
  * group score = sum of the `group_topk` (=2) largest biased affinities in
    the group, added in descending order in fp32;
  * ties go to the lower group index, then to the lower expert index; the K
    outputs of a token are ordered by (biased affinity desc, index asc);
  * expert FFN = SwiGLU without biases: W2 (silu(W1 v) * (W3 v));
  * no residual, gate scale factor 1, dropless;
  * the permutation is expert-major, token-ascending (stable counting sort);
  * bias update: counts_e * E > T*K  ->  b_e -= gamma;  < -> b_e += gamma;
    equal -> unchanged, compared in integers, the add done in fp32;
  * FP8: scale = amax / 448 (fp32 division; 1 when amax == 0), code =
    e4m3(v / scale) with round-to-nearest-even and saturation to +/-448;
    activations in 1x128 tiles along the contraction axis, weights in
    128x128 blocks; each 128-wide block partial product is scaled and summed
    in float64;
  * FP8 with power-of-two scales (the UE8M0 mode, an option beside the
    pages' fp32 scales): scale = the smallest power of two not below
    amax / 448, kept inside UE8M0's range [2^-127, 2^127] (1 when amax == 0);
    codes and GEMMs as above, so only the scale rule differs.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
F64 = np.float64
E4M3_MAX = 448.0


# ----------------------------------------------------------------------------
# Routing  [digest-2.2], [resmic-moe]
# ----------------------------------------------------------------------------

def router_scores(x: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    """Sigmoid token-to-expert affinities s [T, E] (fp32).

    u = x W_r^T is accumulated in float64 and rounded to fp32 (the router is a
    plain linear map [resmic-moe]); s = 1 / (1 + exp(-u)) is evaluated in
    float64 and rounded to fp32 (V3 uses sigmoid, not softmax [digest-2.2]).
    """
    u = (np.asarray(x, F64) @ np.asarray(w_router, F64).T).astype(F32)
    return (1.0 / (1.0 + np.exp(-u.astype(F64)))).astype(F32)


def biased_scores(s: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """s' = s + b, one IEEE fp32 add per element [digest-2.2]."""
    return np.asarray(s, F32) + np.asarray(bias, F32)[None, :]


def group_scores(sp: np.ndarray, G: int, group_topk: int = 2) -> np.ndarray:
    """Score of each of the G groups: sum of its group_topk largest s'.

    The pages choose nodes by the summed affinities of the experts on each
    node [digest-2.2]; the sum runs over the group's group_topk largest
    biased affinities, added largest first in fp32.
    """
    T, E = sp.shape
    per = sp.reshape(T, G, E // G)
    desc = -np.sort(-per, axis=2)  # largest first
    acc = desc[:, :, 0].astype(F32)
    for j in range(1, group_topk):
        acc = (acc + desc[:, :, j]).astype(F32)
    return acc


def select_groups(gs: np.ndarray, M: int) -> np.ndarray:
    """Boolean mask [T, G] of the M groups with the largest score.

    Stable sort on the negated score: equal scores keep index order, so the
    lower group index wins a tie.
    """
    order = np.argsort(-gs, axis=1, kind="stable")[:, :M]
    mask = np.zeros(gs.shape, dtype=bool)
    np.put_along_axis(mask, order, True, axis=1)
    return mask


def select_experts(s: np.ndarray, bias: np.ndarray, G: int, K: int, M: int,
                   group_topk: int = 2):
    """Group-limited top-K routing of each token [digest-2.2].

    Returns (topk_idx int32 [T, K], topk_gate fp32 [T, K]). The selection runs
    on s' = s + b; the gate of a chosen expert is its raw affinity s divided
    by the sum of the raw affinities of the K chosen experts (float64, then
    rounded to fp32), so the bias never enters the gate values.
    """
    s = np.asarray(s, F32)
    T, E = s.shape
    sp = biased_scores(s, bias)
    gmask = select_groups(group_scores(sp, G, group_topk), M)
    emask = np.repeat(gmask, E // G, axis=1)
    cand = np.where(emask, sp, -np.inf).astype(F32)
    idx = np.argsort(-cand, axis=1, kind="stable")[:, :K].astype(np.int32)
    chosen = np.take_along_axis(s, idx, axis=1).astype(F64)
    gate = (chosen / chosen.sum(axis=1, keepdims=True)).astype(F32)
    return idx, gate


# ----------------------------------------------------------------------------
# Load count, scan, permutation  [digest-2.2] (batch load monitoring, dropless)
# ----------------------------------------------------------------------------

def expert_counts(topk_idx: np.ndarray, E: int) -> np.ndarray:
    """counts[e] = number of (token, slot) pairs routed to expert e."""
    return np.bincount(np.asarray(topk_idx).ravel(), minlength=E).astype(np.int32)


def exclusive_offsets(counts: np.ndarray) -> np.ndarray:
    """offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]  (E+1 entries)."""
    out = np.zeros(len(counts) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(counts, np.int64))
    return out.astype(np.int32)


def permutation(topk_idx: np.ndarray, E: int):
    """Expert-major, token-ascending order of all T*K (token, slot) pairs.

    Returns (sorted_tok [T*K] int32, slot_pos [T, K] int32): position p holds
    token sorted_tok[p]; slot k of token t lands at position slot_pos[t, k].
    Written as the definition: experts in ascending order, and inside each
    expert the tokens that chose it in ascending order. Every pair gets a
    position, so no token is dropped.
    """
    idx = np.asarray(topk_idx)
    T, K = idx.shape
    sorted_tok = np.empty(T * K, dtype=np.int32)
    slot_pos = np.full((T, K), -1, dtype=np.int32)
    p = 0
    for e in range(E):
        toks, slots = np.nonzero(idx == e)  # row-major: tokens ascending
        n = len(toks)
        sorted_tok[p:p + n] = toks
        slot_pos[toks, slots] = np.arange(p, p + n, dtype=np.int32)
        p += n
    assert p == T * K
    return sorted_tok, slot_pos


# ----------------------------------------------------------------------------
# Experts  [digest-2.2], [resmic-moe]
# ----------------------------------------------------------------------------

def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(v: np.ndarray, w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """One expert on rows v [n, d]: W2 (silu(W1 v) * (W3 v)), float64.

    w13 [2I, d] holds W1 (rows 0..I-1) then W3 (rows I..2I-1); w2 is [d, I].
    """
    v = np.asarray(v, F64)
    w13 = np.asarray(w13, F64)
    I = w13.shape[0] // 2
    a = v @ w13[:I].T
    b = v @ w13[I:].T
    return (silu(a) * b) @ np.asarray(w2, F64).T


def shared_output(x: np.ndarray, ws13: np.ndarray, ws2: np.ndarray) -> np.ndarray:
    """Sum of the always-on shared experts over the rows of x [resmic-moe]."""
    out = np.zeros((x.shape[0], ws2.shape[1]), dtype=F64)
    for s in range(ws13.shape[0]):
        out += swiglu_ffn(x, ws13[s], ws2[s])
    return out


def routed_output(x: np.ndarray, topk_idx: np.ndarray, topk_gate: np.ndarray,
                  w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """sum_k g_k FFN_{e_k}(x_t) for every row t of x."""
    x = np.asarray(x, F64)
    out = np.zeros((x.shape[0], w2.shape[1]), dtype=F64)
    for e in np.unique(topk_idx):
        rows, slots = np.nonzero(topk_idx == e)
        y = swiglu_ffn(x[rows], w13[e], w2[e])
        out[rows] += np.asarray(topk_gate, F64)[rows, slots][:, None] * y
    return out


def layer_forward(x, w_router, w13, w2, ws13, ws2, bias, G, K, M, group_topk=2,
                  scores=None):
    """The full layer on the rows of x: shared sum + gate-weighted routed sum.

    Returns a dict with scores, topk_idx, topk_gate and out (float64, before
    rounding to the output dtype). No residual is added [resmic-moe].
    """
    s = router_scores(x, w_router) if scores is None else np.asarray(scores, F32)
    idx, gate = select_experts(s, bias, G, K, M, group_topk)
    out = shared_output(x, ws13, ws2) + routed_output(x, idx, gate, w13, w2)
    return {"scores": s, "topk_idx": idx, "topk_gate": gate, "out": out}


# ----------------------------------------------------------------------------
# Auxiliary-loss-free bias update  [digest-2.2]
# ----------------------------------------------------------------------------

def bias_update(counts: np.ndarray, bias: np.ndarray, gamma: float, T: int,
                K: int) -> np.ndarray:
    """One step: overloaded experts get b -= gamma, underloaded b += gamma.

    An expert's load is its count; the target is the mean load T*K/E. The
    comparison counts_e * E vs T * K is done in integers; the add is fp32.
    """
    counts = np.asarray(counts, np.int64)
    E = len(counts)
    b = np.asarray(bias, F32).copy()
    g = F32(gamma)
    lhs = counts * E
    rhs = np.int64(T) * np.int64(K)
    for e in range(E):
        if lhs[e] > rhs:
            b[e] = F32(b[e] - g)
        elif lhs[e] < rhs:
            b[e] = F32(b[e] + g)
    return b


def load_max_over_mean(counts: np.ndarray, T: int, K: int) -> float:
    """Largest expert load divided by the mean load T*K/E."""
    counts = np.asarray(counts, np.int64)
    return float(F32(counts.max() * len(counts) / (T * K)))


def sequence_balance(scores: np.ndarray, topk_idx: np.ndarray, seq_len: int, alpha: float):
    """Sequence-wise balance statistic of the routing [digest-2.2]: the pages
    keep a sequence-level balance loss with a very small weight but print no
    formula; this is the DeepSeek-V3 report's definition (the report the
    pages digest), read forward-only. For each run of seq_len consecutive
    tokens (the last run may be shorter), with L its length, E experts and K
    per token:
        f_i = E / (K L) * #{t : expert i among the K chosen for token t}
        P_i = (1 / L) * sum_t s_{i,t} / sum_j s_{j,t}
        loss = alpha * sum_i f_i P_i
    s are the raw sigmoid affinities, the chosen experts those of topk_idx.
    Returns (loss [n_seq], f [n_seq, E], P [n_seq, E]) in float64.
    """
    s = np.asarray(scores, F64)
    idx = np.asarray(topk_idx)
    T, E = s.shape
    K = idx.shape[1]
    n_seq = (T + seq_len - 1) // seq_len
    loss = np.zeros(n_seq)
    f = np.zeros((n_seq, E))
    P = np.zeros((n_seq, E))
    for q in range(n_seq):
        rows = slice(q * seq_len, min(T, (q + 1) * seq_len))
        L = rows.stop - rows.start
        chosen = np.zeros(E)
        for e in idx[rows].ravel():
            chosen[e] += 1
        f[q] = E / (K * L) * chosen
        P[q] = (s[rows] / s[rows].sum(axis=1, keepdims=True)).sum(axis=0) / L
        loss[q] = alpha * float((f[q] * P[q]).sum())
    return loss, f, P


def bias_balancing_loop(scores: np.ndarray, bias0: np.ndarray, steps: int,
                        gamma: float, G: int, K: int, M: int, group_topk=2):
    """Repeated route -> count -> bias update on fixed scores.

    Returns (list of bias vectors after each step, list of topk_idx,
    list of max/mean load).
    """
    T, E = scores.shape
    b = np.asarray(bias0, F32).copy()
    biases, idxs, loads = [], [], []
    for _ in range(steps):
        idx, _ = select_experts(scores, b, G, K, M, group_topk)
        c = expert_counts(idx, E)
        loads.append(load_max_over_mean(c, T, K))
        b = bias_update(c, b, gamma, T, K)
        idxs.append(idx)
        biases.append(b.copy())
    return biases, idxs, loads


# ----------------------------------------------------------------------------
# FP8 e4m3 with per-tile scales  [digest-3.1]
# ----------------------------------------------------------------------------

def e4m3_value(v: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest e4m3 value (OCP FP8 E4M3 format).

    E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; largest finite value
    448, smallest subnormal 2^-9, no infinities. Round to nearest, ties to
    even; magnitudes beyond 448 saturate to 448. Returns float64 values.
    """
    v = np.asarray(v, F32).astype(F64)
    a = np.abs(v)
    _, ex = np.frexp(a)              # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)       # binade exponent; subnormals share -6
    quantum = np.ldexp(1.0, e - 3)   # 3 mantissa bits
    q = np.rint(a / quantum) * quantum
    q = np.minimum(q, E4M3_MAX)
    return np.where(np.signbit(v), -q, q)


def e4m3_code(v: np.ndarray) -> np.ndarray:
    """The 8-bit e4m3 encoding of e4m3_value(v)."""
    q = e4m3_value(v)
    sign = np.signbit(q).astype(np.uint8) << 7
    a = np.abs(q)
    _, ex = np.frexp(a)
    e = ex - 1
    normal = (a > 0) & (e >= -6)
    exp_field = np.where(normal, e + 7, 0)
    mant = np.where(normal, a / np.ldexp(1.0, np.where(normal, e, 0)) - 1.0,
                    a / 2.0 ** -9 / 8.0)
    mant_field = np.rint(mant * 8).astype(np.int64)
    code = (exp_field.astype(np.int64) << 3) | mant_field
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    """Value of an e4m3 code (0x7f / 0xff are NaN)."""
    c = np.asarray(code, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    mf = c & 0x7
    val = np.where(ef == 0, mf / 8.0 * 2.0 ** -6,
                   (1.0 + mf / 8.0) * np.ldexp(1.0, ef - 7))
    val = np.where((ef == 0xF) & (mf == 0x7), np.nan, val)
    return sign * val


def tile_scale(amax):
    """Scale of one tile: amax / 448 in fp32, or 1 when the tile is all zero."""
    amax = np.asarray(amax, F32)
    sc = (amax / F32(E4M3_MAX)).astype(F32)
    return np.where(amax > 0, sc, F32(1.0)).astype(F32)


def tile_scale_ue8m0(amax):
    """Power-of-two scale of one tile: the smallest 2^e with 2^e >= amax / 448,
    e clamped to [-127, 127] (the exponents a UE8M0 byte can hold), or 1 when
    the tile is all zero. Returned as fp32 values (2^-127 is an fp32
    subnormal, still exact).

    amax / 448 is formed in float64; it is a power of two exactly when amax is
    448 * 2^k (then the float64 quotient is exact), and otherwise lies at
    least one fp32 ulp away from every power of two, far beyond the float64
    rounding of the quotient, so frexp of the quotient decides e correctly.
    """
    amax = np.asarray(amax, F32).astype(F64)
    r = amax / E4M3_MAX
    m, ex = np.frexp(r)                      # r = m * 2^ex, m in [0.5, 1)
    e = np.where(m == 0.5, ex - 1, ex)       # ceil(log2 r)
    e = np.clip(e, -127, 127)
    sc = np.ldexp(1.0, e).astype(F32)
    return np.where(amax > 0, sc, F32(1.0)).astype(F32)


def _scale_rule(ue8m0: bool):
    return tile_scale_ue8m0 if ue8m0 else tile_scale


def quantize_rows_1x128(v: np.ndarray, ue8m0: bool = False):
    """Per-row 1x128 tiles along the last axis.

    Returns (q values float64 [n, k] (e4m3 grid), scales fp32 [n, ceil(k/128)]).
    q = e4m3(v / scale) with the division done in fp32; the scale follows
    tile_scale, or tile_scale_ue8m0 when ue8m0 is set.
    """
    v = np.asarray(v, F32)
    n, k = v.shape
    nb = (k + 127) // 128
    q = np.empty((n, k), dtype=F64)
    scales = np.empty((n, nb), dtype=F32)
    rule = _scale_rule(ue8m0)
    for b in range(nb):
        blk = v[:, b * 128:(b + 1) * 128]
        sc = rule(np.abs(blk).max(axis=1))
        scales[:, b] = sc
        q[:, b * 128:(b + 1) * 128] = e4m3_value((blk / sc[:, None]).astype(F32))
    return q, scales


def quantize_blocks_128x128(w: np.ndarray, ue8m0: bool = False):
    """128x128 blocks of a [n, k] weight matrix.

    Returns (q values float64 [n, k], scales fp32 [ceil(n/128), ceil(k/128)]).
    The matrix is zero-padded to whole blocks (padding does not change a
    block's amax) and viewed as [n/128, 128, k/128, 128]; each block gets
    scale = amax / 448 (or tile_scale_ue8m0 when ue8m0 is set) and codes
    e4m3(w / scale).
    """
    w = np.asarray(w, F32)
    n, k = w.shape
    nbn, nbk = (n + 127) // 128, (k + 127) // 128
    pad = np.zeros((nbn * 128, nbk * 128), F32)
    pad[:n, :k] = w
    blocks = pad.reshape(nbn, 128, nbk, 128)
    scales = _scale_rule(ue8m0)(np.abs(blocks).max(axis=(1, 3)))
    q = e4m3_value((blocks / scales[:, None, :, None]).astype(F32))
    return q.reshape(nbn * 128, nbk * 128)[:n, :k], scales


def fp8_gemm(qa, sa, qw, sw):
    """C = A W^T from e4m3 tiles: sum over 128-wide K blocks of the block
    product scaled by (row scale of A) * (block scale of W), float64.

    qa [n, k] with sa [n, k/128]; qw [m, k] with sw [m/128, k/128].
    """
    qa = np.asarray(qa, F64)
    qw = np.asarray(qw, F64)
    n, k = qa.shape
    m = qw.shape[0]
    out = np.zeros((n, m), dtype=F64)
    col_block = np.arange(m) // 128
    for b in range((k + 127) // 128):
        part = qa[:, b * 128:(b + 1) * 128] @ qw[:, b * 128:(b + 1) * 128].T
        out += part * np.asarray(sa, F64)[:, b:b + 1] * np.asarray(sw, F64)[col_block, b][None, :]
    return out


def quantize_expert_weights(w13: np.ndarray, w2: np.ndarray, ue8m0: bool = False):
    """128x128 block quantisation of one expert's W13 [2I, d] and W2 [d, I]."""
    q13, s13 = quantize_blocks_128x128(w13, ue8m0)
    q2, s2 = quantize_blocks_128x128(w2, ue8m0)
    return q13, s13, q2, s2


def swiglu_ffn_fp8(qx, sx, q13, s13, q2, s2, ue8m0: bool = False):
    """One expert with e4m3 operands: GEMM1 on (qx, sx) x (q13, s13), SwiGLU in
    float64, h rounded to fp32 and re-quantised in 1x128 tiles along I (with
    the same scale rule as the operands), then GEMM2 on (qh, sh) x (q2, s2)."""
    I = q13.shape[0] // 2
    ab = fp8_gemm(qx, sx, q13, s13)
    h = (silu(ab[:, :I]) * ab[:, I:]).astype(F32)
    qh, sh = quantize_rows_1x128(h, ue8m0)
    return fp8_gemm(qh, sh, q2, s2)


def layer_forward_fp8(x, topk_idx, topk_gate, wq, shared_wq, ue8m0: bool = False):
    """Expert part of the FP8 layer on the rows of x (bf16 values as fp32).

    wq: dict e -> (q13, s13, q2, s2) for the experts that appear in topk_idx;
    shared_wq: list of (q13, s13, q2, s2), one per shared expert. Routing is
    the same as the bf16 layer's (the router GEMM is not in FP8). ue8m0
    selects the power-of-two scale rule for x and h (the weights carry
    theirs already).
    """
    qx, sx = quantize_rows_1x128(np.asarray(x, F32), ue8m0)
    out = np.zeros(np.asarray(x).shape, dtype=F64)  # every expert maps width d back to d
    for (q13, s13, q2, s2) in shared_wq:
        out += swiglu_ffn_fp8(qx, sx, q13, s13, q2, s2, ue8m0)
    for e in np.unique(topk_idx):
        rows, slots = np.nonzero(topk_idx == e)
        y = swiglu_ffn_fp8(qx[rows], sx[rows], *wq[int(e)], ue8m0=ue8m0)
        out[rows] += np.asarray(topk_gate, F64)[rows, slots][:, None] * y
    return out


def layer_forward_fp8_full(x, w_router, w13, w2, ws13, ws2, bias, G, K, M, group_topk=2,
                           ue8m0: bool = False):
    """The FP8 layer on the rows of x: bf16-path routing (router_scores,
    select_experts), then 128x128 block quantisation of the master weights of
    every expert the rows use and of the shared experts, then the e4m3 expert
    path of layer_forward_fp8. w13 / w2 / ws13 / ws2 are indexable stacks of
    per-expert master weights; ue8m0 selects the power-of-two scale rule
    everywhere."""
    s = router_scores(x, w_router)
    idx, gate = select_experts(s, bias, G, K, M, group_topk)
    wq = {int(e): quantize_expert_weights(w13[int(e)], w2[int(e)], ue8m0) for e in np.unique(idx)}
    shared = [quantize_expert_weights(ws13[i], ws2[i], ue8m0) for i in range(ws13.shape[0])]
    out = layer_forward_fp8(np.asarray(x, F32), idx, gate, wq, shared, ue8m0)
    return {"scores": s, "topk_idx": idx, "topk_gate": gate, "out": out}
