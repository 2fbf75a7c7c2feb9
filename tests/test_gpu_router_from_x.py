"""Routing computed from the tokens (moe_route with x and the router weights,
as the layer does): for the affinities that the same call writes out, the
chosen experts, their order, the gates and the load count equal the oracle's
selection on those affinities bit for bit (gates to fp32 rounding)
("DeepSeek-V3技术报告" digest, mpbf.cn, section 2.2); the affinities themselves
match the oracle's sigmoid of the router GEMM to fp32 rounding.

Token counts cover one token, a ragged tile and more rows than one tile per
SM; router weights are random, tied (many equal affinities, so the tie rules
decide), or zero (every affinity 0.5). bf16 routers run bf16 tcgen05 tiles;
fp32 routers run tf32-pair tiles, past 256 experts in two column tiles."""
import numpy as np
import pytest
import torch

from oracle import cpp

pytestmark = pytest.mark.gpu

DEV = "cuda"

SHAPES = [
    # E, G, K, M, gk, act
    (256, 8, 8, 4, 2, "bf16"),    # V3 shape
    (64, 8, 6, 3, 2, "bf16"),     # mid-size layer
    (16, 4, 4, 2, 2, "bf16"),
    (8, 4, 2, 2, 2, "bf16"),
    (96, 6, 5, 2, 3, "bf16"),     # E not a multiple of 32, three-term group score
    (128, 8, 6, 3, 4, "bf16"),    # four-term group score
    (64, 1, 8, 1, 4, "bf16"),     # one group: plain top-K
    (256, 8, 8, 4, 32, "bf16"),   # the plain node sum
    (64, 4, 16, 2, 2, "bf16"),    # K = 16
    (256, 16, 8, 4, 2, "bf16"),   # 16 groups
    (16, 4, 4, 2, 2, "f32"),      # the fp32 layer's routing
    (512, 32, 8, 4, 1, "f32"),    # the largest expert count: two router column tiles
]


def _inputs(T, d, E, kind, seed, dt):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g).to(dt)
    if kind == "random":
        wr = (torch.randn(E, d, generator=g) * 0.05).to(dt)
        b = (torch.randint(-2, 3, (E,), generator=g) / 64.0).float()
    elif kind == "tied":
        base = (torch.randn(3, d, generator=g) * 0.05).to(dt)
        wr = base[torch.arange(E) % 3].contiguous()
        b = torch.zeros(E)
    else:
        wr = torch.zeros(E, d, dtype=dt)
        b = torch.zeros(E)
    return x, wr, b


@pytest.mark.parametrize("E,G,K,M,gk,act", SHAPES)
@pytest.mark.parametrize("kind", ["random", "tied", "zero"])
@pytest.mark.parametrize("T", [1, 300, 20000])
def test_router_selection_on_its_own_scores(E, G, K, M, gk, act, kind, T):
    from mixture_experts_layer_100_b300 import binding as B
    d = 256
    x, wr, b = _inputs(T, d, E, kind, seed=T + E + K, dt=torch.float32 if act == "f32" else torch.bfloat16)
    cfg = B.make_config(T, d, E, G, K, M, 128, 1, gk, act=act)
    ws = B.alloc_workspace(cfg)
    s = torch.full((T, E), float("nan"), device=DEV)
    idx = torch.full((T, K), -7, dtype=torch.int32, device=DEV)
    gate = torch.empty((T, K), dtype=torch.float32, device=DEV)
    counts = torch.full((E,), 123, dtype=torch.int32, device=DEV)
    B.moe_route(cfg, x.to(DEV), wr.to(DEV), None, b.to(DEV), s, idx, gate, counts, ws)
    torch.cuda.synchronize()
    assert B.moe_device_error(ws) == 0
    s = s.cpu().numpy()
    ridx, rgate = cpp.select_experts(s, b.numpy(), G, K, M, gk)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(gate.cpu().numpy(), rgate, rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(counts.cpu().numpy(), cpp.expert_counts(ridx, E))
    # the affinities themselves: sigmoid of the router GEMM to fp32 rounding
    s_ref = cpp.router_scores(x.float().numpy(), wr.float().numpy())
    assert np.abs(s - s_ref).max() < 2e-6
    if kind == "zero":
        assert np.all(s == np.float32(0.5))


def test_router_selection_in_the_layer_matches_moe_route():
    """moe_layer_forward routes the same way: its choices, gates and counts
    equal moe_route's on the same tokens."""
    from mixture_experts_layer_100_b300 import binding as B
    from mixture_experts_layer_100_b300 import synth
    from tests.layer_helpers import device_weights, run_layer
    p = synth.PRESETS["mid_t4096_d2048_e64_bf16"].replace(T=1500, d=256, I=128)
    w = synth.make_weights(p)
    wd = device_weights(w)
    x = synth.make_x(p, w.w_router).to(DEV)
    b = synth.make_bias(p).to(DEV)
    res = run_layer(p, wd, x, b)
    cfg = B.config_from_preset(p)
    ws = B.alloc_workspace(cfg)
    idx = torch.empty((p.T, p.K), dtype=torch.int32, device=DEV)
    gate = torch.empty((p.T, p.K), dtype=torch.float32, device=DEV)
    counts = torch.empty((p.E,), dtype=torch.int32, device=DEV)
    B.moe_route(cfg, x, wd["w_router"], None, b, None, idx, gate, counts, ws)
    torch.cuda.synchronize()
    assert torch.equal(idx, res["topk_idx"]) and torch.equal(gate, res["topk_gate"])
    assert torch.equal(counts, res["counts"])
