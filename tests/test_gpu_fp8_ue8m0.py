"""GPU parity of the FP8 expert path with power-of-two (UE8M0) tile scales,
whose GEMMs scale inside the tensor core (tcgen05 block scaling): the
quantisers bit-exact against the oracle's UE8M0 rule, layer outputs within
6e-2 of the largest oracle output, including inputs whose 1x128 tiles and
128x128 weight blocks span many different scales (a scale read for the
wrong row, block or K step is then off by a power of two)."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_100_b300 import synth
from oracle import moe_oracle as om
from tests.layer_helpers import (DEV, compare, device_weights, oracle_rows_cpp, oracle_rows_fp8,
                                 quantize_device_weights, run_layer, stratified_tokens)

pytestmark = pytest.mark.gpu

BASE = synth.PRESETS["v3_t32768_d7168_e256_fp8_ue8m0"]

SMALL = {
    "t300_d256_e16_i256": dict(T=300, d=256, E=16, G=4, K=4, M=2, I=256, S=1),
    "t515_d512_e32_i384_s2": dict(T=515, d=512, E=32, G=8, K=6, M=3, I=384, S=2),
    "t700_d256_e64_k8_s0": dict(T=700, d=256, E=64, G=8, K=8, M=4, I=128, S=0),
}


def small(name, **kw):
    f = dict(SMALL[name])
    f.update(kw)
    return BASE.replace(name=name, zipf=False, bias="u0.02", steps=1, **f)


def _is_pow2(a: np.ndarray) -> bool:
    return bool(np.all(np.frexp(a.astype(np.float64))[0] == 0.5))


def test_weight_quantizer_ue8m0_bit_exact():
    from mixture_experts_layer_100_b300 import binding as B
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(3, 256, 384, generator=g) * 0.02)
    w[1, :128, 128:256] = 0.0                   # an all-zero block (scale 1)
    w[2, 5, 7] = 300.0                          # one large value
    w[0, 130, 200] = 448.0 * 2.0 ** -6          # block amax exactly 448 * 2^-6
    w = w.to(torch.bfloat16)
    wd = w.to(DEV)
    q = torch.empty(w.shape, dtype=torch.uint8, device=DEV)
    sc = torch.empty((3, 2, 3), dtype=torch.float32, device=DEV)
    B.moe_quantize_weights_e4m3_ue8m0(wd, q, sc)
    torch.cuda.synchronize()
    for m in range(3):
        rq, rs = om.quantize_blocks_128x128(w[m].float().numpy(), ue8m0=True)
        np.testing.assert_array_equal(sc[m].cpu().numpy(), rs)
        np.testing.assert_array_equal(om.e4m3_decode(q[m].cpu().numpy()), rq)
    assert _is_pow2(sc.cpu().numpy())
    assert sc[0, 1, 1].item() == 2.0 ** -6


@pytest.mark.parametrize("T,E,K,d", [(100, 16, 4, 256), (1000, 64, 8, 1024)])
def test_activation_tiles_ue8m0_bit_exact(T, E, K, d):
    from mixture_experts_layer_100_b300 import binding as B
    G = 4 if E == 16 else 8
    cfg = B.make_config(T, d, E, G, K, 2 if E == 16 else 4, 256, 1, 2, act="bf16", expert="e4m3_ue8m0")
    ws = B.alloc_workspace(cfg)
    idx = synth.make_topk_idx(T, E, K, seed=T + 1)
    counts = torch.from_numpy(om.expert_counts(idx.numpy(), E))
    x = (torch.randn(T, d) * 3).to(torch.bfloat16)
    x[3, :128] = 0                              # all-zero tile
    x[4, :128] = 0
    x[4, 17] = 448.0 * 2.0 ** -3                # amax exactly 448 * 2^-3
    x[5, 128:256] *= 2.0 ** -20                 # tiny tile
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    st = torch.empty(T * K, dtype=torch.int32, device=DEV)
    sp = torch.empty(T, K, dtype=torch.int32, device=DEV)
    xp = torch.empty(T * K, d, dtype=torch.uint8, device=DEV)
    xs = torch.empty(d // 128, T * K, dtype=torch.float32, device=DEV)
    B.moe_permute(cfg, idx.to(DEV), counts.to(DEV), off, st, sp, x.to(DEV), xp, xs, ws)
    torch.cuda.synchronize()
    rst, _ = om.permutation(idx.numpy(), E)
    rq, rs = om.quantize_rows_1x128(x.float().numpy()[rst], ue8m0=True)
    np.testing.assert_array_equal(xs.cpu().numpy().T, rs)
    np.testing.assert_array_equal(om.e4m3_decode(xp.cpu().numpy()), rq)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_ue8m0_layer_all_tokens(name):
    p = small(name)
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    wq = quantize_device_weights(device_weights(w), ue8m0=True)
    for k in ("w13", "w2", "ws13", "ws2"):
        if wq[k + "_scale"].numel():
            assert _is_pow2(wq[k + "_scale"].cpu().numpy())
    res = run_layer(p, wq, x.to(DEV), b.to(DEV))
    ref = oracle_rows_fp8(p, w, x, b)
    compare(p, res, ref, b, dtype="e4m3_ue8m0")


def _spread_scales(w: synth.Weights, x: torch.Tensor):
    """Multiply every 128x128 weight block and every 1x128 activation tile
    by its own power of two (2^-3 .. 2^3), so that neighbouring blocks,
    tiles and K steps all carry different scales."""
    for name in ("w13", "w2", "ws13", "ws2"):
        t = getattr(w, name)
        if t.numel() == 0:
            continue
        n, r, c = t.shape
        f = torch.empty(n, (r + 127) // 128, (c + 127) // 128)
        for i in range(f.shape[0]):
            for j in range(f.shape[1]):
                for k in range(f.shape[2]):
                    f[i, j, k] = 2.0 ** ((3 * i + 5 * j + 2 * k) % 7 - 3)
        full = f.repeat_interleave(128, 1).repeat_interleave(128, 2)[:, :r, :c]
        setattr(w, name, (t.float() * full).to(t.dtype))
    T, d = x.shape
    ft = torch.tensor([[2.0 ** ((t + 3 * j) % 7 - 3) for j in range(d // 128)] for t in range(T)])
    return w, (x.float() * ft.repeat_interleave(128, 1)).to(x.dtype)


@pytest.mark.parametrize("mode", ["e4m3", "e4m3_ue8m0"])
@pytest.mark.parametrize("name", ["t300_d256_e16_i256", "t515_d512_e32_i384_s2"])
def test_layer_with_spread_scales(name, mode):
    p = small(name).replace(expert_dtype=mode)
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    w, x = _spread_scales(w, x)
    b = synth.make_bias(p)
    wq = quantize_device_weights(device_weights(w), ue8m0=mode == "e4m3_ue8m0")
    res = run_layer(p, wq, x.to(DEV), b.to(DEV))
    ref = oracle_rows_fp8(p, w, x, b)
    compare(p, res, ref, b, dtype=mode)


def test_ue8m0_entry_points_compose_to_the_layer():
    from mixture_experts_layer_100_b300 import binding as B
    p = small("t515_d512_e32_i384_s2")
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router).to(DEV)
    b0 = synth.make_bias(p).to(DEV)
    wq = quantize_device_weights(device_weights(w), ue8m0=True)
    res = run_layer(p, wq, x, b0.clone(), gamma=p.gamma)
    cfg = B.config_from_preset(p)
    ws = B.alloc_workspace(cfg)
    T, K, E, d = p.T, p.K, p.E, p.d
    idx = torch.empty(T, K, dtype=torch.int32, device=DEV)
    gate = torch.empty(T, K, dtype=torch.float32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    st = torch.empty(T * K, dtype=torch.int32, device=DEV)
    sp = torch.empty(T, K, dtype=torch.int32, device=DEV)
    xp = torch.empty(T * K, d, dtype=torch.uint8, device=DEV)
    xs = torch.empty(d // 128, T * K, dtype=torch.float32, device=DEV)
    yp = torch.empty(T * K, d, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(T, d, dtype=torch.bfloat16, device=DEV)
    weights = B.make_weights(**wq)
    bs = b0.clone()
    B.moe_route(cfg, x, wq["w_router"], None, bs, None, idx, gate, counts, ws)
    B.moe_permute(cfg, idx, counts, off, st, sp, x, xp, xs, ws)
    B.moe_grouped_ffn(cfg, xp, xs, off, weights, yp, ws)
    B.moe_combine(cfg, yp, sp, gate, x, weights, out, ws)
    B.moe_bias_update(cfg, counts, p.gamma, bs)
    torch.cuda.synchronize()
    assert B.moe_device_error(ws) == 0
    assert torch.equal(idx, res["topk_idx"])
    assert torch.equal(out, res["out"])


def test_v3_ue8m0_preset_sampled_tokens():
    """The FP8 preset with power-of-two scales (T = 32768): outputs element by
    element against the C++ oracle's UE8M0 path on a 1024-token sample that
    reaches every expert's first and last permuted row and every tile of the
    three hottest experts."""
    p = BASE
    w = synth.make_weights(p, device=DEV)
    wq = quantize_device_weights(device_weights(w), ue8m0=True)
    x = synth.make_x(p, w.w_router, device=DEV)
    b = synth.make_bias(p)
    res = run_layer(p, wq, x, b.to(DEV), gamma=p.gamma)
    toks = stratified_tokens(res["topk_idx"].cpu().numpy(), p.E, 1024, seed=6)
    compare(p, res, oracle_rows_cpp(p, w, x.cpu(), b, toks, expert_dtype="e4m3_ue8m0"), b, tokens=toks,
            dtype="e4m3_ue8m0", max_flip=0.02)
    assert res["counts"].sum().item() == p.T * p.K
    del w, wq
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [1, 129])
def test_ue8m0_layer_one_token_and_ragged(T):
    """One token (every tile mostly padding) and one row past a whole tile."""
    p = small("t300_d256_e16_i256", T=T)
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    res = run_layer(p, quantize_device_weights(device_weights(w), ue8m0=True), x.to(DEV), b.to(DEV))
    compare(p, res, oracle_rows_fp8(p, w, x, b), b, dtype="e4m3_ue8m0")


def test_ue8m0_all_tokens_on_four_experts():
    """Bias +1 on group 0: four experts take all T = 1000 rows each (eight
    m-tiles per expert, the last one ragged); the others get none."""
    p = small("t300_d256_e16_i256", T=1000)
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = torch.zeros(p.E)
    b[:4] = 1.0
    res = run_layer(p, quantize_device_weights(device_weights(w), ue8m0=True), x.to(DEV), b.to(DEV))
    c = res["counts"].cpu().numpy()
    assert list(c[:4]) == [p.T] * 4 and c[4:].sum() == 0
    compare(p, res, oracle_rows_fp8(p, w, x, b), b, dtype="e4m3_ue8m0")


def test_ue8m0_zero_routed_weights_give_shared_only():
    """All-zero routed weights quantise to all-zero blocks with scale 1; the
    output is the shared experts' FP8 output alone."""
    p = small("t515_d512_e32_i384_s2")
    w = synth.make_weights(p, zero_routed=True)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    wq = quantize_device_weights(device_weights(w), ue8m0=True)
    assert torch.all(wq["w13_scale"] == 1.0) and torch.all(wq["w2_scale"] == 1.0)
    res = run_layer(p, wq, x.to(DEV), b.to(DEV))
    qx, sx = om.quantize_rows_1x128(x.float().numpy(), ue8m0=True)
    shared = sum(om.swiglu_ffn_fp8(qx, sx, *om.quantize_expert_weights(w.ws13[i].float().numpy(),
                                                                      w.ws2[i].float().numpy(), ue8m0=True),
                                   ue8m0=True) for i in range(p.S))
    got = res["out"].float().cpu().numpy()
    assert np.abs(got - shared).max() / np.abs(shared).max() <= 6e-2


def test_ue8m0_empty_batch_is_a_no_op():
    from mixture_experts_layer_100_b300 import binding as B
    p = small("t300_d256_e16_i256", T=0)
    w = synth.make_weights(p.replace(T=1))
    cfg = B.config_from_preset(p)
    ws = B.alloc_workspace(cfg)
    b = torch.zeros(p.E, device=DEV)
    counts = torch.full((p.E,), 5, dtype=torch.int32, device=DEV)
    dummy = torch.empty(16, dtype=torch.int32, device=DEV)
    wq = quantize_device_weights(device_weights(w), ue8m0=True)
    B.moe_layer_forward(cfg, None, B.make_weights(**wq), b, 1e-3, None, dummy, dummy.float(), counts, None, ws)
    torch.cuda.synchronize()
    assert counts.sum().item() == 0 and b.abs().sum().item() == 0
