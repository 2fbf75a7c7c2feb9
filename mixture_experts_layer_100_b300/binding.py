"""Python binding of the C ABI in include/moe.h (argument marshalling only).

Each function has the name of the C entry point it calls and takes torch
tensors (or None for nullable pointers); every step of the layer runs in the
CUDA library. There is no fallback: if libmoe_b300.so is missing or cannot be
loaded, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_b300.so")

MOE_F32, MOE_BF16, MOE_E4M3, MOE_E4M3_UE8M0 = 0, 1, 2, 3
_DT = {"f32": MOE_F32, "bf16": MOE_BF16, "e4m3": MOE_E4M3, "e4m3_ue8m0": MOE_E4M3_UE8M0}

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_DEVICE"}


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


MOE_COMBINE_GATHER, MOE_COMBINE_SCATTER_ADD = 0, 1
_COMBINE = {"gather": MOE_COMBINE_GATHER, "scatter_add": MOE_COMBINE_SCATTER_ADD}


class moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("T", "d", "E", "G", "K", "M", "I", "S", "group_topk", "act", "expert",
                                            "combine")]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_router", "w13", "w2", "ws13", "ws2",
                                               "w13_scale", "w2_scale", "ws13_scale", "ws2_scale")]


def load_library(path: str = _LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run python -m mixture_experts_layer_100_b300.build")
    return ctypes.CDLL(path)


lib = load_library()

_P = ctypes.c_void_p
_SIGS = {
    "moe_workspace_size": [ctypes.POINTER(moe_config), ctypes.POINTER(ctypes.c_size_t)],
    "moe_route": [ctypes.POINTER(moe_config)] + [_P] * 8 + [_P, _P],
    "moe_permute": [ctypes.POINTER(moe_config)] + [_P] * 8 + [_P, _P],
    "moe_grouped_ffn": [ctypes.POINTER(moe_config), _P, _P, _P, ctypes.POINTER(moe_weights), _P, _P, _P],
    "moe_combine": [ctypes.POINTER(moe_config), _P, _P, _P, _P, ctypes.POINTER(moe_weights), _P, _P, _P],
    "moe_bias_update": [ctypes.POINTER(moe_config), _P, ctypes.c_float, _P, _P, _P],
    "moe_layer_forward": [ctypes.POINTER(moe_config), _P, ctypes.POINTER(moe_weights), _P, ctypes.c_float,
                          _P, _P, _P, _P, _P, _P, _P],
    "moe_quantize_weights_e4m3": [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P],
    "moe_quantize_weights_e4m3_ue8m0": [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P],
    "moe_permute_static": [ctypes.POINTER(moe_config)] + [_P] * 7 + [_P],
    "moe_seq_balance": [ctypes.POINTER(moe_config), _P, _P, ctypes.c_int, ctypes.c_float, _P, _P, _P, _P, _P],
    "moe_gather_rows": [_P, ctypes.c_int, _P, ctypes.c_int, ctypes.c_size_t, _P, _P, _P],
    "moe_scatter_rows": [_P, _P, ctypes.c_int, ctypes.c_size_t, _P, ctypes.c_int, _P, _P],
    "moe_set_stage_events": [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int],
    "moe_selftest_timeout": [_P, _P],
    "moe_set_layer_graphs": [ctypes.c_int],
    "moe_layer_graphs_kept": [ctypes.POINTER(ctypes.c_int)],
    "moe_device_error": [_P, _P, ctypes.POINTER(ctypes.c_int)],
    "moe_status_string": [ctypes.c_int],
}
for _name, _args in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_char_p if _name == "moe_status_string" else ctypes.c_int

EXPORTED = tuple(_SIGS)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def make_config(T, d, E, G, K, M, I, S, group_topk=2, act="bf16", expert=None, combine="gather") -> moe_config:
    return moe_config(T, d, E, G, K, M, I, S, group_topk, _DT[act], _DT[expert or act], _COMBINE[combine])


def config_from_preset(p, T: Optional[int] = None, combine: Optional[str] = None) -> moe_config:
    return make_config(p.T if T is None else T, p.d, p.E, p.G, p.K, p.M, p.I, p.S, p.group_topk,
                       p.dtype, p.expert_dtype, combine or p.combine)


def make_weights(w_router=None, w13=None, w2=None, ws13=None, ws2=None, w13_scale=None, w2_scale=None,
                 ws13_scale=None, ws2_scale=None) -> moe_weights:
    return moe_weights(*[_ptr(t) for t in (w_router, w13, w2, ws13, ws2, w13_scale, w2_scale,
                                           ws13_scale, ws2_scale)])


def moe_workspace_size(cfg: moe_config) -> int:
    n = ctypes.c_size_t(0)
    _check("moe_workspace_size", lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def alloc_workspace(cfg: moe_config, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of the size the library asks for."""
    return torch.zeros(max(256, moe_workspace_size(cfg)), dtype=torch.uint8, device=device)


def moe_route(cfg, x, w_router, scores_in, bias, scores_out, topk_idx, topk_gate, counts, ws, stream=None):
    _check("moe_route", lib.moe_route(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(scores_in), _ptr(bias),
                                      _ptr(scores_out), _ptr(topk_idx), _ptr(topk_gate), _ptr(counts), _ptr(ws),
                                      _stream(stream)))


def moe_permute(cfg, topk_idx, counts, offsets, sorted_tok, slot_pos, x, xp, xp_scale, ws, stream=None):
    _check("moe_permute", lib.moe_permute(ctypes.byref(cfg), _ptr(topk_idx), _ptr(counts), _ptr(offsets),
                                          _ptr(sorted_tok), _ptr(slot_pos), _ptr(x), _ptr(xp), _ptr(xp_scale),
                                          _ptr(ws), _stream(stream)))


def moe_permute_static(cfg, topk_idx, counts, offsets, sorted_tok, slot_pos, x, xp, stream=None):
    _check("moe_permute_static", lib.moe_permute_static(ctypes.byref(cfg), _ptr(topk_idx), _ptr(counts),
                                                        _ptr(offsets), _ptr(sorted_tok), _ptr(slot_pos), _ptr(x),
                                                        _ptr(xp), _stream(stream)))


def moe_grouped_ffn(cfg, xp, xp_scale, offsets, weights: moe_weights, yp, ws, stream=None):
    _check("moe_grouped_ffn", lib.moe_grouped_ffn(ctypes.byref(cfg), _ptr(xp), _ptr(xp_scale), _ptr(offsets),
                                                  ctypes.byref(weights), _ptr(yp), _ptr(ws), _stream(stream)))


def moe_combine(cfg, yp, slot_pos, topk_gate, x, weights: moe_weights, out, ws, stream=None):
    _check("moe_combine", lib.moe_combine(ctypes.byref(cfg), _ptr(yp), _ptr(slot_pos), _ptr(topk_gate), _ptr(x),
                                          ctypes.byref(weights), _ptr(out), _ptr(ws), _stream(stream)))


def moe_bias_update(cfg, counts, gamma: float, bias, max_over_mean=None, stream=None):
    _check("moe_bias_update", lib.moe_bias_update(ctypes.byref(cfg), _ptr(counts), ctypes.c_float(gamma),
                                                  _ptr(bias), _ptr(max_over_mean), _stream(stream)))


def moe_layer_forward(cfg, x, weights: moe_weights, bias, gamma: float, out, topk_idx, topk_gate, counts,
                      max_over_mean, ws, stream=None):
    _check("moe_layer_forward", lib.moe_layer_forward(
        ctypes.byref(cfg), _ptr(x), ctypes.byref(weights), _ptr(bias), ctypes.c_float(gamma), _ptr(out),
        _ptr(topk_idx), _ptr(topk_gate), _ptr(counts), _ptr(max_over_mean), _ptr(ws), _stream(stream)))


def moe_quantize_weights_e4m3(w, q, scale, stream=None):
    """w [n_mat, rows, cols] bf16 -> q uint8 (same shape), scale [n_mat, rows/128, cols/128] fp32."""
    n_mat, rows, cols = w.shape
    _check("moe_quantize_weights_e4m3", lib.moe_quantize_weights_e4m3(
        _ptr(w), n_mat, rows, cols, _ptr(q), _ptr(scale), _stream(stream)))


def moe_quantize_weights_e4m3_ue8m0(w, q, scale, stream=None):
    """As moe_quantize_weights_e4m3, with power-of-two (UE8M0) block scales."""
    n_mat, rows, cols = w.shape
    _check("moe_quantize_weights_e4m3_ue8m0", lib.moe_quantize_weights_e4m3_ue8m0(
        _ptr(w), n_mat, rows, cols, _ptr(q), _ptr(scale), _stream(stream)))


def moe_seq_balance(cfg, scores, topk_idx, seq_len: int, alpha: float, loss, f=None, p=None, ws=None,
                    stream=None):
    """Per-run sequence-wise balance statistic; scores None reads the
    affinities left in ws by the last routing call."""
    _check("moe_seq_balance", lib.moe_seq_balance(
        ctypes.byref(cfg), _ptr(scores), _ptr(topk_idx), int(seq_len), ctypes.c_float(alpha), _ptr(loss), _ptr(f),
        _ptr(p), _ptr(ws), _stream(stream)))


def _row_bytes(t: torch.Tensor) -> int:
    return t[0].numel() * t.element_size() if t.shape[0] else t.element_size()


def moe_gather_rows(src, idx, dst, ws, stream=None):
    """dst[i] = src[idx[i]] (rows); idx int32 on the device."""
    _check("moe_gather_rows", lib.moe_gather_rows(_ptr(src), src.shape[0], _ptr(idx), idx.numel(), _row_bytes(dst),
                                                  _ptr(dst), _ptr(ws), _stream(stream)))


def moe_scatter_rows(src, idx, dst, ws, stream=None):
    """dst[idx[i]] = src[i] (rows); idx int32 on the device."""
    _check("moe_scatter_rows", lib.moe_scatter_rows(_ptr(src), _ptr(idx), idx.numel(), _row_bytes(src), _ptr(dst),
                                                    dst.shape[0], _ptr(ws), _stream(stream)))


def moe_set_stage_events(events) -> None:
    """events: list of >= 8 recorded torch.cuda.Event (or None to switch off)."""
    if not events:
        _check("moe_set_stage_events", lib.moe_set_stage_events(None, 0))
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check("moe_set_stage_events", lib.moe_set_stage_events(arr, len(events)))


def moe_set_layer_graphs(enable: bool) -> None:
    """Switch the CUDA-graph replay of moe_layer_forward on or off."""
    _check("moe_set_layer_graphs", lib.moe_set_layer_graphs(1 if enable else 0))


def moe_layer_graphs_kept() -> int:
    n = ctypes.c_int(0)
    _check("moe_layer_graphs_kept", lib.moe_layer_graphs_kept(ctypes.byref(n)))
    return n.value


def moe_selftest_timeout(ws, stream=None) -> None:
    _check("moe_selftest_timeout", lib.moe_selftest_timeout(_ptr(ws), _stream(stream)))


def moe_device_error(ws, stream=None) -> int:
    code = ctypes.c_int(0)
    st = lib.moe_device_error(_ptr(ws), _stream(stream), ctypes.byref(code))
    if st not in (MOE_OK, 4, 5):
        raise MoeError("moe_device_error", st)
    return code.value


def moe_status_string(status: int) -> str:
    return lib.moe_status_string(status).decode()
