"""Host-side checks of the C-ABI library: it loads without a GPU, exports
every entry point that include/moe.h declares, and rejects bad arguments
before queuing any work."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_100_b300 import binding as B
from mixture_experts_layer_100_b300 import synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_bias_update",
              "moe_layer_forward", "moe_workspace_size"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(B._LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(B.EXPORTED)


def test_status_strings():
    assert B.moe_status_string(0) == "ok"
    assert "invalid" in B.moe_status_string(1)
    assert B.moe_status_string(99) == "unknown status"


@pytest.mark.parametrize("name", sorted(synth.PRESETS))
def test_workspace_size_presets(name):
    p = synth.PRESETS[name]
    cfg = B.config_from_preset(p)
    n = B.moe_workspace_size(cfg)
    # at least the permuted rows and the routed outputs
    assert n >= p.T * p.K * p.d * 2


@pytest.mark.parametrize("field,value,status", [
    ("E", 15, 1),          # E % G != 0
    ("M", 5, 1),           # M > G
    ("K", 9, 1),           # K > M * E / G  (E=16, G=4, M=2)
    ("group_topk", 5, 1),  # group_topk > E / G
    ("G", 64, 1),          # E % G
    ("E", 1024, 2),        # more experts than the library supports (G divides)
    ("T", -1, 1),
])
def test_invalid_configs(field, value, status):
    cfg = B.make_config(T=8, d=512, E=16, G=4, K=4, M=2, I=256, S=1, act="f32")
    setattr(cfg, field, value)
    if field == "E" and value == 1024:
        cfg.G = 32
    n = ctypes.c_size_t(0)
    assert B.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == status


def test_bf16_shape_limits():
    cfg = B.make_config(T=8, d=200, E=16, G=4, K=4, M=2, I=256, S=1, act="bf16")
    n = ctypes.c_size_t(0)
    assert B.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == 2
    cfg = B.make_config(T=8, d=256, E=16, G=4, K=4, M=2, I=256, S=1, act="f32", expert="e4m3")
    assert B.lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == 1


def test_null_pointers_rejected_before_any_cuda_call():
    cfg = B.make_config(T=8, d=512, E=16, G=4, K=4, M=2, I=256, S=1, act="f32")
    st = B.lib.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None, None)
    assert st == 1
    st = B.lib.moe_bias_update(ctypes.byref(cfg), None, ctypes.c_float(1e-3), None, None, None)
    assert st == 1
    w = B.moe_weights()
    st = B.lib.moe_layer_forward(ctypes.byref(cfg), None, ctypes.byref(w), None, ctypes.c_float(0), None, None,
                                 None, None, None, None, None)
    assert st == 1
    # misaligned pointer
    st = B.lib.moe_bias_update(ctypes.byref(cfg), ctypes.c_void_p(0x1004), ctypes.c_float(1e-3),
                               ctypes.c_void_p(0x2000), None, None)
    assert st == 1


def test_newer_entry_points_reject_bad_arguments_before_any_cuda_call():
    cfg = B.make_config(T=8, d=512, E=16, G=4, K=4, M=2, I=256, S=1, act="f32")
    f = ctypes.c_float
    # sequence-wise balance statistic: seq_len must be positive; indices and loss are required
    assert B.lib.moe_seq_balance(ctypes.byref(cfg), ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), 0, f(1.0),
                                 ctypes.c_void_p(0x3000), None, None, None, None) == 1
    assert B.lib.moe_seq_balance(ctypes.byref(cfg), ctypes.c_void_p(0x1000), None, 4, f(1.0),
                                 ctypes.c_void_p(0x3000), None, None, None, None) == 1
    assert B.lib.moe_seq_balance(ctypes.byref(cfg), ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), 4, f(1.0),
                                 None, None, None, None, None) == 1
    # scores taken from the workspace need a workspace
    assert B.lib.moe_seq_balance(ctypes.byref(cfg), None, ctypes.c_void_p(0x2000), 4, f(1.0),
                                 ctypes.c_void_p(0x3000), None, None, None, None) == 1
    # misaligned f / p outputs
    assert B.lib.moe_seq_balance(ctypes.byref(cfg), ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), 4, f(1.0),
                                 ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4002), None, None, None) == 1
    # T = 0: nothing to do
    cfg0 = B.make_config(T=0, d=512, E=16, G=4, K=4, M=2, I=256, S=1, act="f32")
    assert B.lib.moe_seq_balance(ctypes.byref(cfg0), None, None, 4, f(1.0), None, None, None, None, None) == 0
    # weight quantisers: negative sizes, missing buffers; empty is a no-op
    for q in (B.lib.moe_quantize_weights_e4m3, B.lib.moe_quantize_weights_e4m3_ue8m0):
        assert q(ctypes.c_void_p(0x1000), -1, 128, 128, ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), None) == 1
        assert q(None, 1, 128, 128, ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), None) == 1
        assert q(ctypes.c_void_p(0x1000), 1, 128, 128, ctypes.c_void_p(0x2000), None, None) == 1
        assert q(None, 0, 128, 128, None, None, None) == 0
    # stage-event hook: off is fine, fewer than 8 events or a null array is not
    assert B.lib.moe_set_stage_events(None, 0) == 0
    assert B.lib.moe_set_stage_events(None, 8) == 1
    arr = (ctypes.c_void_p * 4)(*([0x10] * 4))
    assert B.lib.moe_set_stage_events(arr, 4) == 1
    arr8 = (ctypes.c_void_p * 8)(*([0x10] * 7 + [None]))
    assert B.lib.moe_set_stage_events(arr8, 8) == 1
    # graph replay toggle: on / off only
    assert B.lib.moe_set_layer_graphs(2) == 1
    assert B.lib.moe_set_layer_graphs(0) == 0 and B.lib.moe_set_layer_graphs(1) == 0
    assert B.lib.moe_layer_graphs_kept(None) == 1 and B.moe_layer_graphs_kept() == 0
    # device error query needs a workspace and an output
    code = ctypes.c_int(0)
    assert B.lib.moe_device_error(None, None, ctypes.byref(code)) == 1
    assert B.lib.moe_device_error(ctypes.c_void_p(0x1000), None, None) == 1
