"""GPU parity of routing, load count, permutation and bias update.

Both sides get identical inputs from the seeded generators (fp32 affinity
scores, expert choices, bias); indices, counts, offsets, permutation and the
bias trajectory must match the oracle bit for bit, gates to fp32 rounding.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_100_b300 import synth
from oracle import moe_oracle as om

pytestmark = pytest.mark.gpu

DEV = "cuda"


def B():
    from mixture_experts_layer_100_b300 import binding
    return binding


def _route_gpu(cfg, s, b, ws=None):
    Bn = B()
    T, E = s.shape
    K = cfg.K
    idx = torch.full((T, K), -7, dtype=torch.int32, device=DEV)
    gate = torch.empty((T, K), dtype=torch.float32, device=DEV)
    counts = torch.full((E,), 123, dtype=torch.int32, device=DEV)
    ws = Bn.alloc_workspace(cfg) if ws is None else ws
    Bn.moe_route(cfg, None, None, s.to(DEV), b.to(DEV), None, idx, gate, counts, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), gate.cpu().numpy(), counts.cpu().numpy()


ROUTE_SHAPES = [
    # E, G, K, M, gk
    (16, 4, 4, 2, 2),     # tiny fp32 layer
    (64, 8, 6, 3, 2),     # mid-size bf16 layer
    (256, 8, 8, 4, 2),    # V3 shape
    (8, 4, 2, 2, 2),
    (96, 6, 5, 2, 3),     # E not a multiple of 32, three-term group score
    (512, 32, 8, 4, 1),   # the largest supported expert count
    (64, 4, 6, 2, 16),    # group score = plain sum over the group (the pages' node score)
    (256, 8, 8, 4, 32),   # V3 shape with the plain node sum
    (64, 4, 16, 2, 2),    # K = 16
    (128, 4, 32, 4, 2),   # K = 32, the largest the library takes
]


@pytest.mark.parametrize("E,G,K,M,gk", ROUTE_SHAPES)
@pytest.mark.parametrize("kind", ["uniform", "dyadic", "const", "skewed"])
@pytest.mark.parametrize("T", [1, 37, 1000])
def test_route_identical_scores(E, G, K, M, gk, kind, T):
    Bn = B()
    s = synth.make_scores(T, E, seed=T + E, kind=kind)
    rng = np.random.default_rng(E + K)
    b = torch.from_numpy(((rng.integers(-3, 4, E) / 32.0) if kind == "dyadic"
                          else rng.uniform(-0.02, 0.02, E)).astype(np.float32))
    cfg = Bn.make_config(T, 128, E, G, K, M, 128, 1, gk, act="bf16" if E <= 256 else "f32")
    idx, gate, counts = _route_gpu(cfg, s, b)
    ridx, rgate = om.select_experts(s.numpy(), b.numpy(), G, K, M, gk)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(gate, rgate, rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(counts, om.expert_counts(ridx, E))


@pytest.mark.parametrize("name", ["tiny_t256_d512_e16_fp32", "mid_t4096_d2048_e64_bf16",
                                  "v3_t16384_d7168_e256_bf16", "v3_decode_t64_bf16",
                                  "v3_t32768_d7168_e256_fp8"])
def test_route_full_size_presets(name):
    """Routing of every preset at its full token count, on identical scores."""
    Bn = B()
    p = synth.PRESETS[name]
    s = synth.make_scores(p.T, p.E, seed=1, kind="skewed")
    b = synth.make_bias(p)
    cfg = Bn.config_from_preset(p)
    idx, gate, counts = _route_gpu(cfg, s, b)
    ridx, rgate = om.select_experts(s.numpy(), b.numpy(), p.G, p.K, p.M, p.group_topk)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(gate, rgate, rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(counts, om.expert_counts(ridx, p.E))


def test_route_golden_two_tokens():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "two_token_example.json")))
    Bn = B()
    s = torch.tensor(g["scores"], dtype=torch.float32)
    b = torch.tensor(g["bias"], dtype=torch.float32)
    cfg = Bn.make_config(2, 128, g["E"], g["G"], g["K"], g["M"], 128, 1, g["group_topk"], act="f32")
    idx, gate, counts = _route_gpu(cfg, s, b)
    np.testing.assert_array_equal(idx, g["topk_idx"])
    np.testing.assert_array_equal(counts, g["counts"])
    want = np.array([[n / d for n, d in r] for r in g["topk_gate_num_den"]], np.float32)
    np.testing.assert_array_equal(gate, want)
    # permutation and bias update of the same example
    ws = Bn.alloc_workspace(cfg)
    x = torch.arange(2 * 128, dtype=torch.float32, device=DEV).reshape(2, 128)
    off = torch.empty(g["E"] + 1, dtype=torch.int32, device=DEV)
    st = torch.empty(4, dtype=torch.int32, device=DEV)
    sp = torch.empty(2, 2, dtype=torch.int32, device=DEV)
    xp = torch.empty(4, 128, dtype=torch.float32, device=DEV)
    Bn.moe_permute(cfg, torch.tensor(idx, device=DEV), torch.tensor(counts, device=DEV), off, st, sp, x, xp,
                   None, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(off.cpu().numpy(), g["offsets"])
    np.testing.assert_array_equal(st.cpu().numpy(), g["sorted_tok"])
    np.testing.assert_array_equal(sp.cpu().numpy(), g["slot_pos"])
    bd = b.to(DEV)
    Bn.moe_bias_update(cfg, torch.tensor(counts, device=DEV), g["gamma"], bd)
    want_b = om.bias_update(np.array(g["counts"]), b.numpy(), g["gamma"], 2, g["K"])
    np.testing.assert_array_equal(bd.cpu().numpy(), want_b)
    assert np.array_equal(np.sign(bd.cpu().numpy() - b.numpy()), g["bias_delta_sign"])


@pytest.mark.parametrize("T,E,K,d,act", [(1, 16, 4, 512, "f32"), (37, 16, 4, 512, "f32"),
                                         (1000, 64, 6, 256, "bf16"), (4096, 64, 6, 2048, "bf16"),
                                         (16384, 256, 8, 7168, "bf16"), (77, 256, 8, 128, "bf16")])
def test_permute_identical_choices(T, E, K, d, act):
    Bn = B()
    idx = synth.make_topk_idx(T, E, K, seed=T)
    counts = om.expert_counts(idx.numpy(), E)
    G = 4 if E == 16 else 8
    cfg = Bn.make_config(T, d, E, G, K, 2 if E == 16 else 4, 128, 1, 2, act=act)
    ws = Bn.alloc_workspace(cfg)
    dt = torch.float32 if act == "f32" else torch.bfloat16
    x = torch.randn(T, d, device=DEV).to(dt)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    st = torch.empty(T * K, dtype=torch.int32, device=DEV)
    sp = torch.empty(T, K, dtype=torch.int32, device=DEV)
    xp = torch.empty(T * K, d, dtype=dt, device=DEV)
    Bn.moe_permute(cfg, idx.to(DEV), torch.from_numpy(counts).to(DEV), off, st, sp, x, xp, None, ws)
    torch.cuda.synchronize()
    assert Bn.moe_device_error(ws) == 0
    rst, rsp = om.permutation(idx.numpy(), E)
    np.testing.assert_array_equal(off.cpu().numpy(), om.exclusive_offsets(counts))
    np.testing.assert_array_equal(st.cpu().numpy(), rst)
    np.testing.assert_array_equal(sp.cpu().numpy(), rsp)
    assert torch.equal(xp, x[torch.from_numpy(rst).long().to(DEV)])


def test_permute_reports_bad_expert_index():
    """An expert index outside [0, E) is skipped and flagged, not followed."""
    Bn = B()
    T, E, K, d = 64, 16, 4, 128
    idx = synth.make_topk_idx(T, E, K, seed=3)
    idx[5, 2] = E + 3
    counts = torch.from_numpy(om.expert_counts(np.clip(idx.numpy(), 0, E - 1), E))
    cfg = Bn.make_config(T, d, E, 4, K, 2, 128, 1, 2, act="f32")
    ws = Bn.alloc_workspace(cfg)
    x = torch.randn(T, d, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    st = torch.zeros(T * K, dtype=torch.int32, device=DEV)
    sp = torch.zeros(T, K, dtype=torch.int32, device=DEV)
    xp = torch.zeros(T * K, d, device=DEV)
    Bn.moe_permute(cfg, idx.to(DEV), counts.to(DEV), off, st, sp, x, xp, None, ws)
    code = Bn.moe_device_error(ws)
    assert code in (0x201, 0x202)
    assert Bn.moe_device_error(ws) == 0  # read clears it


@pytest.mark.parametrize("name,steps,T", [("tiny_t256_d512_e16_fp32", 10, None),
                                          ("v3_t32768_d7168_e256_fp8", 50, None),
                                          ("mid_t4096_d2048_e64_bf16", 20, None)])
def test_bias_trajectory_bit_exact(name, steps, T):
    """route -> count -> bias update repeated on fixed scores: indices, bias
    and max/mean load every step equal the oracle's."""
    Bn = B()
    p = synth.PRESETS[name]
    T = p.T if T is None else T
    s = synth.make_scores(T, p.E, seed=5, kind="skewed")
    b0 = synth.make_bias(p)
    cfg = Bn.config_from_preset(p, T=T)
    ws = Bn.alloc_workspace(cfg)
    sd, bd = s.to(DEV), b0.clone().to(DEV)
    idx = torch.empty(T, p.K, dtype=torch.int32, device=DEV)
    gate = torch.empty(T, p.K, dtype=torch.float32, device=DEV)
    counts = torch.empty(p.E, dtype=torch.int32, device=DEV)
    mom = torch.empty(1, dtype=torch.float32, device=DEV)
    biases, idxs, loads = om.bias_balancing_loop(s.numpy(), b0.numpy(), steps, p.gamma, p.G, p.K, p.M,
                                                 p.group_topk)
    for i in range(steps):
        Bn.moe_route(cfg, None, None, sd, bd, None, idx, gate, counts, ws)
        Bn.moe_bias_update(cfg, counts, p.gamma, bd, mom)
        np.testing.assert_array_equal(idx.cpu().numpy(), idxs[i])
        np.testing.assert_array_equal(bd.cpu().numpy(), biases[i])
        assert mom.item() == loads[i]
    assert loads[-1] < loads[0]


def test_device_wait_gives_up_and_reports_timeout():
    """A wait on a barrier that nothing releases returns after about a second
    with a timeout code; the context stays usable afterwards."""
    import time
    Bn = B()
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    t0 = time.time()
    Bn.moe_selftest_timeout(ws)
    code = Bn.moe_device_error(ws)
    assert code == 0x105 and time.time() - t0 < 30
    assert Bn.moe_device_error(ws) == 0
    # the GPU still runs work
    s = synth.make_scores(64, 16, seed=9)
    cfg = Bn.make_config(64, 128, 16, 4, 4, 2, 128, 1, 2, act="f32")
    idx, _, _ = _route_gpu(cfg, s, torch.zeros(16))
    np.testing.assert_array_equal(idx, om.select_experts(s.numpy(), np.zeros(16, np.float32), 4, 4, 2)[0])
