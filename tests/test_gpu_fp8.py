"""GPU parity of the FP8 expert path (e4m3 GEMM inputs with 1x128 activation
tiles and 128x128 weight blocks, fp32 accumulation): quantisers bit-exact,
layer outputs within 6e-2 of the largest oracle output."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_100_b300 import synth
from oracle import moe_oracle as om
from tests.layer_helpers import (DEV, compare, device_weights, oracle_rows_cpp, oracle_rows_fp8,
                                 quantize_device_weights, run_layer, stratified_tokens)

pytestmark = pytest.mark.gpu

BASE = synth.PRESETS["v3_t32768_d7168_e256_fp8"]

SMALL = {
    "t300_d256_e16_i256": dict(T=300, d=256, E=16, G=4, K=4, M=2, I=256, S=1),
    "t515_d512_e32_i384_s2": dict(T=515, d=512, E=32, G=8, K=6, M=3, I=384, S=2),
    "t700_d256_e64_k8_s0": dict(T=700, d=256, E=64, G=8, K=8, M=4, I=128, S=0),
}


def small(name, **kw):
    f = dict(SMALL[name])
    f.update(kw)
    return BASE.replace(name=name, zipf=False, bias="u0.02", steps=1, **f)


def test_weight_quantizer_bit_exact():
    from mixture_experts_layer_100_b300 import binding as B
    g = torch.Generator().manual_seed(3)
    w = (torch.randn(3, 256, 384, generator=g) * 0.02)
    w[1, :128, 128:256] = 0.0                   # an all-zero block (scale 1)
    w[2, 5, 7] = 300.0                          # one large value
    w = w.to(torch.bfloat16)
    wd = w.to(DEV)
    q = torch.empty(w.shape, dtype=torch.uint8, device=DEV)
    sc = torch.empty((3, 2, 3), dtype=torch.float32, device=DEV)
    B.moe_quantize_weights_e4m3(wd, q, sc)
    torch.cuda.synchronize()
    for m in range(3):
        rq, rs = om.quantize_blocks_128x128(w[m].float().numpy())
        np.testing.assert_array_equal(sc[m].cpu().numpy(), rs)
        np.testing.assert_array_equal(om.e4m3_decode(q[m].cpu().numpy()), rq)


@pytest.mark.parametrize("T,E,K,d", [(100, 16, 4, 256), (1000, 64, 8, 1024)])
def test_activation_tiles_in_permute_bit_exact(T, E, K, d):
    from mixture_experts_layer_100_b300 import binding as B
    G = 4 if E == 16 else 8
    cfg = B.make_config(T, d, E, G, K, 2 if E == 16 else 4, 256, 1, 2, act="bf16", expert="e4m3")
    ws = B.alloc_workspace(cfg)
    idx = synth.make_topk_idx(T, E, K, seed=T)
    counts = torch.from_numpy(om.expert_counts(idx.numpy(), E))
    x = (torch.randn(T, d) * 3).to(torch.bfloat16)
    x[3, :128] = 0  # all-zero tile
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    st = torch.empty(T * K, dtype=torch.int32, device=DEV)
    sp = torch.empty(T, K, dtype=torch.int32, device=DEV)
    xp = torch.empty(T * K, d, dtype=torch.uint8, device=DEV)
    xs = torch.empty(d // 128, T * K, dtype=torch.float32, device=DEV)
    B.moe_permute(cfg, idx.to(DEV), counts.to(DEV), off, st, sp, x.to(DEV), xp, xs, ws)
    torch.cuda.synchronize()
    rst, _ = om.permutation(idx.numpy(), E)
    rq, rs = om.quantize_rows_1x128(x.float().numpy()[rst])
    np.testing.assert_array_equal(xs.cpu().numpy().T, rs)
    np.testing.assert_array_equal(om.e4m3_decode(xp.cpu().numpy()), rq)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_fp8_layer_all_tokens(name):
    p = small(name)
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router)
    b = synth.make_bias(p)
    wq = quantize_device_weights(device_weights(w))
    res = run_layer(p, wq, x.to(DEV), b.to(DEV))
    ref = oracle_rows_fp8(p, w, x, b)
    compare(p, res, ref, b, dtype="e4m3")


def test_fp8_entry_points_compose_to_the_layer():
    from mixture_experts_layer_100_b300 import binding as B
    p = small("t515_d512_e32_i384_s2")
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router).to(DEV)
    b0 = synth.make_bias(p).to(DEV)
    wq = quantize_device_weights(device_weights(w))
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


@pytest.fixture(scope="module")
def v3_fp8():
    p = BASE
    w = synth.make_weights(p, device=DEV)
    wq = quantize_device_weights(device_weights(w))
    yield p, w, wq
    del w, wq
    torch.cuda.empty_cache()


def test_v3_fp8_preset_sampled_tokens(v3_fp8):
    """The FP8 preset (T = 32768): outputs element by element against the C++
    oracle's e4m3 path on a 1024-token sample that reaches every expert's
    first and last permuted row and every tile of the three hottest experts."""
    p, w, wq = v3_fp8
    x = synth.make_x(p, w.w_router, device=DEV)
    b = synth.make_bias(p)
    res = run_layer(p, wq, x, b.to(DEV), gamma=p.gamma)
    toks = stratified_tokens(res["topk_idx"].cpu().numpy(), p.E, 1024, seed=4)
    compare(p, res, oracle_rows_cpp(p, w, x.cpu(), b, toks, expert_dtype="e4m3"), b, tokens=toks, dtype="e4m3",
            max_flip=0.02)
    assert res["counts"].sum().item() == p.T * p.K
