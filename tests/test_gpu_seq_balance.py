"""GPU parity of the sequence-wise balance statistic (f, P and the loss per
run of seq_len tokens) against the oracle on identical scores and choices."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_100_b300 import synth
from oracle import moe_oracle as om

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(cfg, s, idx, seq_len, alpha, ws=None, scores_from_ws=False):
    from mixture_experts_layer_100_b300 import binding as B
    n = (cfg.T + seq_len - 1) // seq_len
    loss = torch.full((n,), float("nan"), device=DEV)
    f = torch.full((n, cfg.E), float("nan"), device=DEV)
    p = torch.full((n, cfg.E), float("nan"), device=DEV)
    B.moe_seq_balance(cfg, None if scores_from_ws else s, idx, seq_len, alpha, loss, f, p, ws)
    torch.cuda.synchronize()
    return loss.cpu().numpy(), f.cpu().numpy(), p.cpu().numpy()


@pytest.mark.parametrize("T,E,K,seq_len", [(1, 16, 4, 4096), (300, 16, 4, 128), (4096, 64, 6, 1000),
                                           (16384, 256, 8, 4096), (5000, 512, 8, 1700), (777, 96, 5, 1)])
def test_seq_balance_identical_inputs(T, E, K, seq_len):
    from mixture_experts_layer_100_b300 import binding as B
    s = synth.make_scores(T, E, seed=T + 5, kind="uniform")
    idx = synth.make_topk_idx(T, E, K, seed=T + 6)
    cfg = B.make_config(T, 128, E, 4 if E % 4 == 0 else 1, K, 4 if E % 4 == 0 else 1, 128, 1, 1,
                        act="f32")
    loss, f, p = _run(cfg, s.to(DEV), idx.to(DEV), seq_len, 1e-3)
    rl, rf, rp = om.sequence_balance(s.numpy(), idx.numpy(), seq_len, 1e-3)
    np.testing.assert_allclose(f, rf, rtol=1e-6)
    np.testing.assert_allclose(p, rp, rtol=2e-5, atol=1e-9)
    np.testing.assert_allclose(loss, rl, rtol=2e-5)


def test_seq_balance_reads_scores_left_by_routing():
    """scores = NULL uses the affinities the routing call left in the
    workspace; the result is bit-identical to passing them explicitly, and
    matches the oracle on those scores and choices."""
    from mixture_experts_layer_100_b300 import binding as B
    p_ = synth.PRESETS["mid_t4096_d2048_e64_bf16"]
    w = synth.make_weights(p_, device=DEV)
    x = synth.make_x(p_, w.w_router, device=DEV)
    cfg = B.config_from_preset(p_)
    ws = B.alloc_workspace(cfg)
    T, E, K = p_.T, p_.E, p_.K
    scores = torch.empty(T, E, device=DEV)
    idx = torch.empty(T, K, dtype=torch.int32, device=DEV)
    gate = torch.empty(T, K, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    bias = synth.make_bias(p_, device=DEV)
    B.moe_route(cfg, x, w.w_router, None, bias, scores, idx, gate, counts, ws)
    a = _run(cfg, scores, idx, 1024, 1e-4)
    B.moe_route(cfg, x, w.w_router, None, bias, None, idx, gate, counts, ws)
    b = _run(cfg, None, idx, 1024, 1e-4, ws=ws, scores_from_ws=True)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
    rl, rf, rp = om.sequence_balance(scores.cpu().numpy(), idx.cpu().numpy(), 1024, 1e-4)
    np.testing.assert_allclose(a[0], rl, rtol=2e-5)
    np.testing.assert_allclose(a[1], rf, rtol=1e-6)


def test_seq_balance_deterministic():
    from mixture_experts_layer_100_b300 import binding as B
    T, E, K = 8192, 256, 8
    s = synth.make_scores(T, E, seed=9, kind="skewed").to(DEV)
    idx = synth.make_topk_idx(T, E, K, seed=10).to(DEV)
    cfg = B.make_config(T, 128, E, 8, K, 4, 128, 1, 2, act="bf16")
    r1 = _run(cfg, s, idx, 2048, 0.5)
    r2 = _run(cfg, s, idx, 2048, 0.5)
    for u, v in zip(r1, r2):
        np.testing.assert_array_equal(u, v)
