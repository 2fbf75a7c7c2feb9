"""GPU parity of the whole layer (moe_layer_forward) and of the individual
entry points, against the oracle on the same seeded inputs.

Small shapes are compared element by element on every token; they span
several 128-row tiles per expert, ragged tails, both down-projection tile
widths, S = 0 / 1 / 2 shared experts and the degenerate cases (one token,
all-tied router, zero routed weights, all tokens on a few experts, T = 0).
The full-size presets: routing of every token bit-exact given the library's
own affinities, outputs element by element on seeded samples of at least 1024
tokens that reach every expert (all tokens for the mid-size and decode
shapes).
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_100_b300 import synth
from oracle import moe_oracle as om
from tests.layer_helpers import (DEV, compare, device_weights, oracle_rows, oracle_rows_cpp, run_layer,
                                 stratified_tokens)

pytestmark = pytest.mark.gpu

BASE = synth.PRESETS["mid_t4096_d2048_e64_bf16"]

SMALL = {
    "t300_d256_e16_i256": dict(T=300, d=256, E=16, G=4, K=4, M=2, I=256, S=1),
    "t515_d384_e32_i384_s2": dict(T=515, d=384, E=32, G=8, K=6, M=3, I=384, S=2),
    "t1_d256_e16": dict(T=1, d=256, E=16, G=4, K=4, M=2, I=128, S=1),
    "t700_d128_e256_k8": dict(T=700, d=128, E=256, G=8, K=8, M=4, I=128, S=1),
    "t129_d512_e64_s0": dict(T=129, d=512, E=64, G=8, K=6, M=3, I=256, S=0),
    "t200_d256_e128_k6": dict(T=200, d=256, E=128, G=8, K=6, M=3, I=128, S=1),
    "t333_d256_e32_nodesum": dict(T=333, d=256, E=32, G=4, K=4, M=2, I=128, S=1, group_topk=8),
    "t150_d256_e64_k16": dict(T=150, d=256, E=64, G=4, K=16, M=2, I=128, S=1),
    "t90_d256_e64_k32": dict(T=90, d=256, E=64, G=2, K=32, M=1, I=128, S=1),
    "t257_d256_e32_k1": dict(T=257, d=256, E=32, G=4, K=1, M=1, I=128, S=1),   # top-1 routing, one group
    # T * K >= 128 E: the bf16 layer uses the zero-padded expert layout
    "t520_d256_e8_padded": dict(T=520, d=256, E=8, G=4, K=2, M=2, I=128, S=1),
}


def small_preset(name, **over):
    kw = dict(SMALL[name])
    kw.update(over)
    return BASE.replace(name=name, zipf=False, bias="u0.01", **kw)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("combine", ["gather", "scatter_add"])
@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_layer_all_tokens(name, combine, dtype):
    """bf16 layers, and fp32 layers (tf32-pair tensor-core GEMMs, 1e-5)."""
    p = small_preset(name, combine=combine, dtype=dtype, expert_dtype=dtype)
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    res = run_layer(p, device_weights(w), x.to(DEV), b.to(DEV))
    ref = oracle_rows(p, w, x, b)
    compare(p, res, ref, b)
    np.testing.assert_array_equal(res["counts"].cpu().numpy(),
                                  om.expert_counts(res["topk_idx"].cpu().numpy(), p.E))


def test_tiny_fp32_preset_with_bias_steps():
    """The fp32 preset: full output parity at 1e-5, then its 10 forward +
    bias-update steps; the bias trajectory must equal the oracle's."""
    p = synth.PRESETS["tiny_t256_d512_e16_fp32"]
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    wd = device_weights(w)
    xd, bd = x.to(DEV), b.clone().to(DEV)
    b_ref = b.numpy().copy()
    ws = None
    for step in range(p.steps):
        res = run_layer(p, wd, xd, bd, gamma=p.gamma, ws=ws)
        ws = res["ws"]
        ref = oracle_rows(p, w, x, torch.from_numpy(b_ref))
        compare(p, res, ref, b_ref, max_flip=0.0)
        b_ref = om.bias_update(om.expert_counts(ref["topk_idx"], p.E), b_ref, p.gamma, p.T, p.K)
        np.testing.assert_array_equal(bd.cpu().numpy(), b_ref)


@pytest.mark.parametrize("combine", ["gather", "scatter_add"])
def test_fp32_layer_with_512_experts(combine):
    """The largest expert count (fp32 layers only): the router runs two
    256-column tiles and the grouped GEMMs walk 512 groups."""
    p = small_preset("t300_d256_e16_i256", T=400, d=128, E=512, G=32, K=8, M=4, I=128, S=1, combine=combine,
                     dtype="f32", expert_dtype="f32")
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    res = run_layer(p, device_weights(w), x.to(DEV), b.to(DEV))
    compare(p, res, oracle_rows(p, w, x, b), b)
    assert res["counts"].sum().item() == p.T * p.K


@pytest.mark.parametrize("combine", ["gather", "scatter_add"])
def test_all_tokens_on_four_experts(combine):
    """Bias +1 on group 0: every token takes its four experts (4 x T rows)."""
    p = small_preset("t300_d256_e16_i256", T=1000, combine=combine)
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = torch.zeros(p.E)
    b[:4] = 1.0
    res = run_layer(p, device_weights(w), x.to(DEV), b.to(DEV))
    c = res["counts"].cpu().numpy()
    assert list(c[:4]) == [p.T] * 4 and c[4:].sum() == 0
    compare(p, res, oracle_rows(p, w, x, b), b)


def test_zero_router_all_ties():
    p = small_preset("t300_d256_e16_i256")
    w = synth.make_weights(p)
    w.w_router.zero_()
    x = synth.make_x(p, w.w_router)
    b = torch.zeros(p.E)
    res = run_layer(p, device_weights(w), x.to(DEV), b.to(DEV))
    idx = res["topk_idx"].cpu().numpy()
    assert (idx == np.arange(4)[None, :]).all()
    assert (res["topk_gate"].cpu().numpy() == np.float32(0.25)).all()
    compare(p, res, oracle_rows(p, w, x, b), b)


@pytest.mark.parametrize("combine", ["gather", "scatter_add"])
def test_zero_routed_weights_give_shared_only(combine):
    p = small_preset("t515_d384_e32_i384_s2", combine=combine)
    w = synth.make_weights(p, zero_routed=True)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    res = run_layer(p, device_weights(w), x.to(DEV), b.to(DEV))
    shared = om.shared_output(x.double().numpy(), w.ws13.double().numpy(), w.ws2.double().numpy())
    got = res["out"].float().cpu().numpy()
    assert np.abs(got - shared).max() / np.abs(shared).max() <= 2e-2


def test_empty_batch_is_a_no_op():
    from mixture_experts_layer_100_b300 import binding as B
    p = small_preset("t300_d256_e16_i256", T=0)
    w = synth.make_weights(p.replace(T=1))
    cfg = B.config_from_preset(p)
    ws = B.alloc_workspace(cfg)
    b = torch.zeros(p.E, device=DEV)
    counts = torch.full((p.E,), 5, dtype=torch.int32, device=DEV)
    dummy = torch.empty(16, dtype=torch.int32, device=DEV)
    B.moe_layer_forward(cfg, None, B.make_weights(**device_weights(w)), b, 1e-3, None, dummy, dummy.float(),
                        counts, None, ws)
    torch.cuda.synchronize()
    assert counts.sum().item() == 0 and b.abs().sum().item() == 0


@pytest.mark.parametrize("name", ["t515_d384_e32_i384_s2", "t520_d256_e8_padded"])
def test_entry_points_compose_to_the_layer(name):
    """route -> permute -> grouped_ffn -> combine -> bias_update gives the
    same bits as moe_layer_forward (for t520 the layer runs its experts on the
    zero-padded row layout, the entry points on contiguous rows)."""
    from mixture_experts_layer_100_b300 import binding as B
    p = small_preset(name)
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router).to(DEV)
    b0 = synth.make_bias(p).to(DEV)
    wd = device_weights(w)
    bl = b0.clone()
    res = run_layer(p, wd, x, bl, gamma=p.gamma)
    cfg = B.config_from_preset(p)
    ws = B.alloc_workspace(cfg)
    T, K, E, d = p.T, p.K, p.E, p.d
    idx = torch.empty(T, K, dtype=torch.int32, device=DEV)
    gate = torch.empty(T, K, dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    scores = torch.empty(T, E, dtype=torch.float32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    st = torch.empty(T * K, dtype=torch.int32, device=DEV)
    sp = torch.empty(T, K, dtype=torch.int32, device=DEV)
    xp = torch.empty(T * K, d, dtype=torch.bfloat16, device=DEV)
    yp = torch.empty(T * K, d, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(T, d, dtype=torch.bfloat16, device=DEV)
    weights = B.make_weights(**wd)
    bs = b0.clone()
    B.moe_route(cfg, x, wd["w_router"], None, bs, scores, idx, gate, counts, ws)
    B.moe_permute(cfg, idx, counts, off, st, sp, x, xp, None, ws)
    B.moe_grouped_ffn(cfg, xp, None, off, weights, yp, ws)
    B.moe_combine(cfg, yp, sp, gate, x, weights, out, ws)
    B.moe_bias_update(cfg, counts, p.gamma, bs)
    torch.cuda.synchronize()
    assert B.moe_device_error(ws) == 0
    assert torch.equal(idx, res["topk_idx"]) and torch.equal(counts, res["counts"])
    assert torch.equal(out, res["out"])
    assert torch.equal(bs, bl)
    # the router scores: sigmoid(x W_r^T) to fp32 rounding of the bf16 GEMM
    s_ref = om.router_scores(x.float().cpu().numpy(), w.w_router.float().numpy())
    assert np.abs(scores.cpu().numpy() - s_ref).max() < 2e-6
    # and the routed rows themselves: yp[p] = FFN_e(x[sorted_tok[p]])
    o = off.cpu().numpy()
    for e in [0, 7, E - 1]:
        rows = np.arange(o[e], o[e + 1])[:5]
        if len(rows) == 0:
            continue
        toks = st.cpu().numpy()[rows]
        ref = om.swiglu_ffn(x.float().cpu().numpy()[toks], w.w13[e].double().numpy(), w.w2[e].double().numpy())
        got = yp[torch.from_numpy(rows).to(DEV)].float().cpu().numpy()
        assert np.abs(got - ref).max() / np.abs(ref).max() <= 2e-2


def test_scatter_add_combine_matches_gather():
    """The two combine modes compute the same sums in a different order: they
    agree to fp32 rounding of K gated rows (before the bf16 output rounding),
    and the routing, loads and bias are identical."""
    p = small_preset("t515_d384_e32_i384_s2")
    w = synth.make_weights(p)
    wd = device_weights(w)
    x = synth.make_x(p, w.w_router).to(DEV)
    b0 = synth.make_bias(p).to(DEV)
    bg, bs = b0.clone(), b0.clone()
    rg = run_layer(p, wd, x, bg, gamma=p.gamma)
    rs = run_layer(p.replace(combine="scatter_add"), wd, x, bs, gamma=p.gamma)
    for k in ("topk_idx", "topk_gate", "counts"):
        assert torch.equal(rg[k], rs[k])
    assert torch.equal(bg, bs)
    og, os_ = rg["out"].float(), rs["out"].float()
    assert (og - os_).abs().max().item() <= 2 ** -7 * og.abs().max().item()


def test_layer_is_deterministic():
    p = small_preset("t515_d384_e32_i384_s2")
    w = synth.make_weights(p)
    wd = device_weights(w)
    x = synth.make_x(p, w.w_router).to(DEV)
    b = synth.make_bias(p).to(DEV)
    r1 = run_layer(p, wd, x, b)
    r2 = run_layer(p, wd, x, b)
    assert torch.equal(r1["out"], r2["out"]) and torch.equal(r1["topk_idx"], r2["topk_idx"])


def test_mid_preset_all_tokens():
    p = synth.PRESETS["mid_t4096_d2048_e64_bf16"]
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    res = run_layer(p, device_weights(w), x.to(DEV), b.to(DEV))
    compare(p, res, oracle_rows(p, w, x, b), b)
    assert res["counts"].sum().item() == p.T * p.K


def gpu_scores(p, wd, x, b):
    """The affinities the library's router computes for x (moe_route with
    scores_out); the router GEMM is deterministic, so every layer call on the
    same x routes on exactly these values."""
    from mixture_experts_layer_100_b300 import binding as B
    cfg = B.config_from_preset(p)
    ws = B.alloc_workspace(cfg)
    s = torch.empty(p.T, p.E, dtype=torch.float32, device=DEV)
    idx = torch.empty(p.T, p.K, dtype=torch.int32, device=DEV)
    gate = torch.empty(p.T, p.K, dtype=torch.float32, device=DEV)
    counts = torch.empty(p.E, dtype=torch.int32, device=DEV)
    B.moe_route(cfg, x, wd["w_router"], None, b, s, idx, gate, counts, ws)
    torch.cuda.synchronize()
    assert B.moe_device_error(ws) == 0
    return s.cpu().numpy(), idx, gate, counts


@pytest.fixture(scope="module")
def v3_weights():
    p = synth.PRESETS["v3_t16384_d7168_e256_bf16"]
    w = synth.make_weights(p, device=DEV)
    torch.cuda.synchronize()
    yield w
    del w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("combine", ["gather", "scatter_add"])
def test_v3_preset_full_size(v3_weights, combine):
    """The bench workload (T = 16384, V3 shape, skewed routing): routing of
    every token bit-exact against the oracle given the library's own scores,
    and the layer output element by element on a 1024-token sample that
    reaches every expert's first and last permuted row and every tile of the
    three hottest experts."""
    from oracle import cpp
    p = synth.PRESETS["v3_t16384_d7168_e256_bf16"].replace(combine=combine)
    w = v3_weights
    x = synth.make_x(p, w.w_router, device=DEV)
    b = synth.make_bias(p)
    wd = device_weights(w)
    res = run_layer(p, wd, x, b.to(DEV), gamma=p.gamma)
    s, idx_r, gate_r, counts_r = gpu_scores(p, wd, x, b.to(DEV))
    idx_ref, gate_ref = cpp.select_experts(s, b.numpy(), p.G, p.K, p.M, p.group_topk)
    idx = res["topk_idx"].cpu().numpy()
    np.testing.assert_array_equal(idx, idx_ref)
    np.testing.assert_array_equal(idx_r.cpu().numpy(), idx_ref)
    np.testing.assert_allclose(res["topk_gate"].cpu().numpy(), gate_ref, rtol=2e-6)
    c = res["counts"].cpu().numpy()
    np.testing.assert_array_equal(c, cpp.expert_counts(idx_ref, p.E))
    assert res["max_over_mean"].item() == cpp.load_max_over_mean(c, p.T, p.K)
    toks = stratified_tokens(idx, p.E, 1024, seed=1)
    assert len(toks) >= 1024
    compare(p, res, oracle_rows_cpp(p, w, x.cpu(), b, toks), b, tokens=toks)
    # skewed raw load: the hottest expert well above the mean
    assert c.max() > 4 * c.mean()


@pytest.mark.parametrize("name", ["v3_decode_t64_bf16", "v3_decode_t512_bf16"])
def test_v3_decode_presets_all_tokens(v3_weights, name):
    p = synth.PRESETS[name]
    w = v3_weights
    x = synth.make_x(p, w.w_router, device=DEV)
    b = synth.make_bias(p)
    res = run_layer(p, device_weights(w), x, b.to(DEV))
    compare(p, res, oracle_rows_cpp(p, w, x.cpu(), b), b, max_flip=0.02)


def test_bias_checkpoint_resumes_bit_exactly():
    """The layer's only state is the routing bias: saving it after 3 steps and
    resuming from the saved copy gives the same trajectory as 6 straight steps."""
    from mixture_experts_layer_100_b300 import state
    p = small_preset("t300_d256_e16_i256")
    w = synth.make_weights(p)
    wd = device_weights(w)
    x = synth.make_x(p, w.w_router).to(DEV)
    b_run = synth.make_bias(p).to(DEV)
    for _ in range(6):
        run_layer(p, wd, x, b_run, gamma=p.gamma)
    b_a = synth.make_bias(p).to(DEV)
    for _ in range(3):
        run_layer(p, wd, x, b_a, gamma=p.gamma)
    blob = state.save_bias(b_a, step=3)
    b_b, step = state.load_bias(blob, device=DEV)
    assert step == 3
    for _ in range(3):
        run_layer(p, wd, x, b_b, gamma=p.gamma)
    assert torch.equal(b_b, b_run)


def test_fp8_preset_balancing_loop_on_the_layer():
    """The FP8 preset's loop on the full layer: 50 forward + bias-update steps
    on fixed inputs. Given the library's own affinities, the chosen experts,
    the bias and the max/mean load of every step equal the oracle's
    bias-balancing loop bit for bit; the peak load comes down."""
    from oracle import cpp
    from tests.layer_helpers import quantize_device_weights
    p = synth.PRESETS["v3_t32768_d7168_e256_fp8"]
    w = synth.make_weights(p, device=DEV)
    wq = quantize_device_weights(device_weights(w))
    del w
    x = synth.make_x(p, wq["w_router"], device=DEV)
    b0 = synth.make_bias(p)
    b = b0.clone().to(DEV)
    s, _, _, _ = gpu_scores(p, wq, x, b)
    biases, idxs, loads = cpp.bias_balancing_loop(s, b0.numpy(), p.steps, p.gamma, p.G, p.K, p.M, p.group_topk)
    from mixture_experts_layer_100_b300 import binding as B
    ws = B.alloc_workspace(B.config_from_preset(p))
    for step in range(p.steps):
        res = run_layer(p, wq, x, b, gamma=p.gamma, ws=ws)
        np.testing.assert_array_equal(res["topk_idx"].cpu().numpy(), idxs[step])
        np.testing.assert_array_equal(b.cpu().numpy(), biases[step])
        assert res["max_over_mean"].item() == loads[step]
        assert res["counts"].sum().item() == p.T * p.K
    assert loads[-1] < loads[0], (loads[0], loads[-1])
