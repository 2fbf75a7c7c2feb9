"""moe_permute_static: the permutation for callers that cannot allocate device
memory (code handed only its input and output buffers, or running under a
fixed memory budget). It must give exactly what moe_permute gives with a
workspace, call after call, although every call reuses one static scratch
array; and it must refuse a batch too large for that array.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_100_b300 import synth
from oracle import moe_oracle as om

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _both(T, E, K, d, seed):
    from mixture_experts_layer_100_b300 import binding as B
    G = 8 if E % 8 == 0 else 4
    cfg = B.make_config(T, d, E, G, K, 4 if E % 8 == 0 else 2, 128, 1, 2, act="bf16")
    idx = synth.make_topk_idx(T, E, K, seed=seed).to(DEV)
    counts = torch.from_numpy(om.expert_counts(idx.cpu().numpy(), E)).to(DEV)
    x = torch.randn(T, d, device=DEV).to(torch.bfloat16)

    def bufs():
        return (torch.full((E + 1,), -1, dtype=torch.int32, device=DEV),
                torch.full((T * K,), -1, dtype=torch.int32, device=DEV),
                torch.full((T, K), -1, dtype=torch.int32, device=DEV),
                torch.zeros(T * K, d, dtype=torch.bfloat16, device=DEV))

    ref = bufs()
    ws = B.alloc_workspace(cfg)
    B.moe_permute(cfg, idx, counts, *ref[:3], x, ref[3], None, ws)
    got = bufs()
    st = B.lib.moe_permute_static(ctypes.byref(cfg), B._ptr(idx), B._ptr(counts), B._ptr(got[0]),
                                  B._ptr(got[1]), B._ptr(got[2]), B._ptr(x), B._ptr(got[3]),
                                  B._stream(None))
    assert st == 0, B.moe_status_string(st)
    torch.cuda.synchronize()
    # integer outputs and copied rows: bit-exact, the tolerance of the permutation tests
    for a, b in zip(ref, got):
        assert torch.equal(a, b)
    return got


def test_static_scratch_permute_matches_workspace_version():
    # several calls in a row, small / large / small, through the one static array
    _both(1000, 64, 6, 256, seed=1)
    _both(16384, 256, 8, 512, seed=2)
    got = _both(37, 16, 4, 128, seed=3)
    st, sp = om.permutation(synth.make_topk_idx(37, 16, 4, seed=3).numpy(), 16)
    np.testing.assert_array_equal(got[1].cpu().numpy(), st)
    np.testing.assert_array_equal(got[2].cpu().numpy(), sp)


def test_static_scratch_permute_rejects_oversized_batch():
    from mixture_experts_layer_100_b300 import binding as B
    T, E, K = 65536, 256, 8  # needs 256 + 2 MiB + 4 MiB > 4 MiB
    cfg = B.make_config(T, 128, E, 8, K, 4, 128, 1, 2, act="bf16")
    dummy = torch.empty(64, dtype=torch.int32, device=DEV)
    p = B._ptr(dummy)
    st = B.lib.moe_permute_static(ctypes.byref(cfg), p, p, p, p, p, p, p, B._stream(None))
    assert st == 2  # MOE_ERR_UNSUPPORTED, nothing queued


def test_static_scratch_permute_allocates_nothing():
    """Calls after the first one leave the device's free memory and torch's
    reserved pool exactly as they were (the scratch is the static array, not
    a new allocation), and the Python binding of the entry point gives the
    same bits as the C call."""
    from mixture_experts_layer_100_b300 import binding as B
    T, E, K, d = 4096, 64, 6, 256
    cfg = B.make_config(T, d, E, 8, K, 3, 128, 1, 2, act="bf16")
    idx = synth.make_topk_idx(T, E, K, seed=7).to(DEV)
    counts = torch.from_numpy(om.expert_counts(idx.cpu().numpy(), E)).to(DEV)
    x = torch.randn(T, d, device=DEV).to(torch.bfloat16)
    outs = [(torch.empty(E + 1, dtype=torch.int32, device=DEV), torch.empty(T * K, dtype=torch.int32, device=DEV),
             torch.empty(T, K, dtype=torch.int32, device=DEV), torch.empty(T * K, d, dtype=torch.bfloat16, device=DEV))
            for _ in range(2)]
    B.moe_permute_static(cfg, idx, counts, *outs[0][:3], x, outs[0][3])  # first call: module loaded, address looked up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for i in range(3):
        o = outs[i % 2]
        B.moe_permute_static(cfg, idx, counts, *o[:3], x, o[3])
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_reserved() == reserved0
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    st, sp = om.permutation(idx.cpu().numpy(), E)
    np.testing.assert_array_equal(outs[0][1].cpu().numpy(), st)
    np.testing.assert_array_equal(outs[0][2].cpu().numpy(), sp)
