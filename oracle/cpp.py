"""ctypes wrapper of the C++ CPU oracle (libmoe_oracle.so, oracle/moe_oracle.h).

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's CPU
legs import this module. It converts numpy arrays to the C types the oracle
takes and back; every step of the layer runs in the C++ library, which is
the plain definition of the layer ("DeepSeek-V3技术报告" digest, mpbf.cn,
sections 2.2 and 3.1; "DeepSeek-V3架构深度解析", blog.resmic.cn, 核心架构二).
The library is built on first import if it is missing or older than its
source.
"""
from __future__ import annotations

import ctypes

import numpy as np

from oracle import build as _build

_lib = ctypes.CDLL(_build.build())

_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
_u8 = ctypes.c_uint8
_i = ctypes.c_int
_l = ctypes.c_int64
_vp = ctypes.c_void_p

_SIGS = {
    "mo_hardware_threads": ([], _i),
    "mo_router_scores": ([_f32p, _l, _i, _f32p, _i, _i, _f32p], None),
    "mo_select_experts": ([_f32p, _f32p, _l, _i, _i, _i, _i, _i, _i, _i32p, _f32p], None),
    "mo_group_scores": ([_f32p, _f32p, _l, _i, _i, _i, _f32p], None),
    "mo_expert_counts": ([_i32p, _l, _i, _i, _i32p], None),
    "mo_exclusive_offsets": ([_i32p, _i, _i32p], None),
    "mo_permutation": ([_i32p, _l, _i, _i, _i32p, _i32p], None),
    "mo_bias_update": ([_i32p, _i, _l, _i, ctypes.c_float, _f32p], None),
    "mo_load_max_over_mean": ([_i32p, _i, _l, _i], ctypes.c_float),
    "mo_bias_balancing_loop": ([_f32p, _f32p, _l, _i, _i, _i, _i, _i, _i, ctypes.c_float, _i, _f32p, _i32p,
                                _f32p], None),
    "mo_swiglu_ffn": ([_f32p, _l, _i, _i, _f32p, _f32p, _i, _f64p], None),
    "mo_expert_accumulate": ([_f32p, _i, _i64p, _l, _i, _f32p, _f32p, _vp, _i, _f64p], None),
    "mo_layer_forward": ([_f32p, _l, _i, _i, _i, _i, _i, _i, _i, _i, _f32p, _f32p, _f32p, _vp, _vp, _f32p, _vp,
                          _i, _f32p, _i32p, _f32p, _f64p], None),
    "mo_e4m3_value": ([ctypes.c_float], ctypes.c_double),
    "mo_e4m3_code": ([ctypes.c_float], _u8),
    "mo_e4m3_decode": ([_u8], ctypes.c_double),
    "mo_tile_scale": ([ctypes.c_float, _i], ctypes.c_float),
    "mo_quantize_rows_1x128": ([_f32p, _l, _i, _i, _f64p, _f32p], None),
    "mo_quantize_blocks_128x128": ([_f32p, _l, _i, _i, _f64p, _f32p], None),
    "mo_fp8_gemm": ([_f64p, _f32p, _l, _i, _f64p, _f32p, _l, _i, _f64p], None),
    "mo_expert_accumulate_fp8": ([_f32p, _i, _i64p, _l, _i, _f32p, _f32p, _vp, _i, _i, _f64p], None),
    "mo_layer_forward_fp8": ([_f32p, _l, _i, _i, _i, _i, _i, _i, _i, _i, _f32p, _f32p, _f32p, _vp, _vp, _f32p,
                              _i, _i, _f32p, _i32p, _f32p, _f64p], None),
    "mo_sequence_balance": ([_f32p, _i32p, _l, _i, _i, _i, ctypes.c_double, _f64p, _vp, _vp], None),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _opt(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def hardware_threads() -> int:
    return int(_lib.mo_hardware_threads())


def router_scores(x, w_router, threads=0):
    x, w = _f32(x), _f32(w_router)
    T, d = x.shape
    E = w.shape[0]
    s = np.empty((T, E), np.float32)
    _lib.mo_router_scores(x, T, d, w, E, threads, s)
    return s


def select_experts(s, bias, G, K, M, group_topk=2, threads=0):
    s = _f32(s)
    T, E = s.shape
    idx = np.empty((T, K), np.int32)
    gate = np.empty((T, K), np.float32)
    _lib.mo_select_experts(s, _f32(bias), T, E, G, K, M, group_topk, threads, idx, gate)
    return idx, gate


def group_scores(s, bias, G, group_topk=2):
    s = _f32(s)
    T, E = s.shape
    gs = np.empty((T, G), np.float32)
    _lib.mo_group_scores(s, _f32(bias), T, E, G, group_topk, gs)
    return gs


def expert_counts(idx, E):
    idx = _i32(idx)
    T, K = idx.shape
    c = np.empty(E, np.int32)
    _lib.mo_expert_counts(idx, T, K, E, c)
    return c


def exclusive_offsets(counts):
    counts = _i32(counts)
    o = np.empty(len(counts) + 1, np.int32)
    _lib.mo_exclusive_offsets(counts, len(counts), o)
    return o


def permutation(idx, E):
    idx = _i32(idx)
    T, K = idx.shape
    st = np.empty(T * K, np.int32)
    sp = np.empty((T, K), np.int32)
    _lib.mo_permutation(idx, T, K, E, st, sp)
    return st, sp


def bias_update(counts, bias, gamma, T, K):
    b = _f32(bias).copy()
    counts = _i32(counts)
    _lib.mo_bias_update(counts, len(counts), T, K, gamma, b)
    return b


def load_max_over_mean(counts, T, K):
    counts = _i32(counts)
    return float(_lib.mo_load_max_over_mean(counts, len(counts), T, K))


def bias_balancing_loop(s, bias0, steps, gamma, G, K, M, group_topk=2, threads=0):
    """Returns (biases [steps, E], idx [steps, T, K], loads [steps])."""
    s = _f32(s)
    T, E = s.shape
    biases = np.empty((steps, E), np.float32)
    idx = np.empty((steps, T, K), np.int32)
    loads = np.empty(steps, np.float32)
    _lib.mo_bias_balancing_loop(s, _f32(bias0), T, E, G, K, M, group_topk, steps, gamma, threads, biases, idx, loads)
    return biases, idx, loads


def swiglu_ffn(v, w13, w2, threads=0):
    v = _f32(v)
    n, d = v.shape
    I = w13.shape[0] // 2
    y = np.empty((n, d), np.float64)
    _lib.mo_swiglu_ffn(v, n, d, I, _f32(w13), _f32(w2), threads, y)
    return y


def expert_accumulate(x, rows, w13, w2, gates, acc, threads=0, fp8=False, ue8m0=False):
    """acc[rows[i]] += gates[i] * FFN(x[rows[i]]) (gates None: 1); rows distinct.
    x [n, d] fp32, acc [n, d] float64 (updated in place)."""
    x = _f32(x)
    assert acc.dtype == np.float64 and acc.flags.c_contiguous and acc.shape[1] == x.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert len(np.unique(rows)) == len(rows)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < min(x.shape[0], acc.shape[0]))
    g = None if gates is None else _f32(gates)
    I = w13.shape[0] // 2
    d = x.shape[1]
    if fp8:
        _lib.mo_expert_accumulate_fp8(x, d, rows, len(rows), I, _f32(w13), _f32(w2), _opt(g), int(ue8m0), threads,
                                      acc)
    else:
        _lib.mo_expert_accumulate(x, d, rows, len(rows), I, _f32(w13), _f32(w2), _opt(g), threads, acc)


def layer_forward(x, w_router, w13, w2, ws13, ws2, bias, G, K, M, group_topk=2, scores=None, threads=0):
    """The full layer on the rows of x (weights as whole stacks in memory).
    Returns dict(scores, topk_idx, topk_gate, out float64)."""
    x = _f32(x)
    T, d = x.shape
    E, I2, _ = w13.shape
    S = ws13.shape[0]
    w13_, w2_ = _f32(w13), _f32(w2)
    ws13_ = _f32(ws13) if S else None
    ws2_ = _f32(ws2) if S else None
    sin = None if scores is None else _f32(scores)
    s = np.empty((T, E), np.float32)
    idx = np.empty((T, K), np.int32)
    gate = np.empty((T, K), np.float32)
    out = np.empty((T, d), np.float64)
    _lib.mo_layer_forward(x, T, d, E, G, K, M, group_topk, I2 // 2, S, _f32(w_router), w13_, w2_, _opt(ws13_),
                          _opt(ws2_), _f32(bias), _opt(sin), threads, s, idx, gate, out)
    return {"scores": s, "topk_idx": idx, "topk_gate": gate, "out": out}


def layer_forward_fp8(x, w_router, w13, w2, ws13, ws2, bias, G, K, M, group_topk=2, ue8m0=False, threads=0):
    x = _f32(x)
    T, d = x.shape
    E, I2, _ = w13.shape
    S = ws13.shape[0]
    ws13_ = _f32(ws13) if S else None
    ws2_ = _f32(ws2) if S else None
    s = np.empty((T, E), np.float32)
    idx = np.empty((T, K), np.int32)
    gate = np.empty((T, K), np.float32)
    out = np.empty((T, d), np.float64)
    _lib.mo_layer_forward_fp8(x, T, d, E, G, K, M, group_topk, I2 // 2, S, _f32(w_router), _f32(w13), _f32(w2),
                              _opt(ws13_), _opt(ws2_), _f32(bias), int(ue8m0), threads, s, idx, gate, out)
    return {"scores": s, "topk_idx": idx, "topk_gate": gate, "out": out}


def e4m3_value(v: float) -> float:
    return float(_lib.mo_e4m3_value(float(v)))


def e4m3_code(v: float) -> int:
    return int(_lib.mo_e4m3_code(float(v)))


def e4m3_decode(c: int) -> float:
    return float(_lib.mo_e4m3_decode(int(c)))


def tile_scale(amax: float, ue8m0: bool = False) -> float:
    return float(_lib.mo_tile_scale(float(amax), int(ue8m0)))


def quantize_rows_1x128(v, ue8m0=False):
    v = _f32(v)
    n, k = v.shape
    q = np.empty((n, k), np.float64)
    sc = np.empty((n, (k + 127) // 128), np.float32)
    _lib.mo_quantize_rows_1x128(v, n, k, int(ue8m0), q, sc)
    return q, sc


def quantize_blocks_128x128(w, ue8m0=False):
    w = _f32(w)
    n, k = w.shape
    q = np.empty((n, k), np.float64)
    sc = np.empty(((n + 127) // 128, (k + 127) // 128), np.float32)
    _lib.mo_quantize_blocks_128x128(w, n, k, int(ue8m0), q, sc)
    return q, sc


def fp8_gemm(qa, sa, qw, sw, threads=0):
    qa = np.ascontiguousarray(qa, np.float64)
    qw = np.ascontiguousarray(qw, np.float64)
    n, k = qa.shape
    m = qw.shape[0]
    out = np.empty((n, m), np.float64)
    _lib.mo_fp8_gemm(qa, _f32(sa), n, k, qw, _f32(sw), m, threads, out)
    return out


def sequence_balance(scores, topk_idx, seq_len, alpha):
    s = _f32(scores)
    idx = _i32(topk_idx)
    T, E = s.shape
    K = idx.shape[1]
    n_seq = (T + seq_len - 1) // seq_len
    loss = np.empty(n_seq, np.float64)
    f = np.empty((n_seq, E), np.float64)
    P = np.empty((n_seq, E), np.float64)
    _lib.mo_sequence_balance(s, idx, T, E, K, seq_len, alpha, loss, f.ctypes.data_as(ctypes.c_void_p),
                             P.ctypes.data_as(ctypes.c_void_p))
    return loss, f, P
