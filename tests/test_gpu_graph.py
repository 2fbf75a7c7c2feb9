"""moe_layer_forward captured into a CUDA graph: replaying the graph gives
bit-for-bit the outputs, expert choices, loads and bias updates of the same
calls made eagerly (the layer's kernels are deterministic; with the
scatter-add combine the output to the last bf16 bit), with the side stream of
the shared experts forked and joined inside the graph."""
import pytest
import torch

from mixture_experts_layer_100_b300 import synth
from tests.layer_helpers import DEV, device_weights, quantize_device_weights

pytestmark = pytest.mark.gpu


def _buffers(p):
    return {
        "out": torch.full((p.T, p.d), float("nan"), dtype=synth.torch_dtype(p.dtype), device=DEV),
        "idx": torch.empty((p.T, p.K), dtype=torch.int32, device=DEV),
        "gate": torch.empty((p.T, p.K), dtype=torch.float32, device=DEV),
        "counts": torch.empty((p.E,), dtype=torch.int32, device=DEV),
        "mom": torch.empty(1, dtype=torch.float32, device=DEV),
    }


def _call(B, cfg, x, W, bias, gamma, o, ws):
    B.moe_layer_forward(cfg, x, W, bias, gamma, o["out"], o["idx"], o["gate"], o["counts"], o["mom"], ws)


@pytest.mark.parametrize("name,expert", [("mid_t4096_d2048_e64_bf16", None),
                                         ("mid_t4096_d2048_e64_bf16_scatter", "scatter_add"),
                                         ("t515_d512_e32_s2_ue8m0", "e4m3_ue8m0"),
                                         ("t515_d512_e32_s2_e4m3", "e4m3"),
                                         ("t300_d256_e16_f32", "f32")])
def test_graph_replay_matches_eager_steps(name, expert):
    from mixture_experts_layer_100_b300 import binding as B
    if name in ("t515_d512_e32_s2_ue8m0", "t515_d512_e32_s2_e4m3"):
        base = "v3_t32768_d7168_e256_fp8_ue8m0" if expert == "e4m3_ue8m0" else "v3_t32768_d7168_e256_fp8"
        p = synth.PRESETS[base].replace(
            name=name, T=515, d=512, E=32, G=8, K=6, M=3, I=384, S=2, zipf=False, bias="u0.02")
    elif name == "t300_d256_e16_f32":
        p = synth.PRESETS["tiny_t256_d512_e16_fp32"].replace(name=name, T=300, d=256, bias="u0.02")
    elif expert == "scatter_add":
        p = synth.PRESETS["mid_t4096_d2048_e64_bf16"].replace(name=name, combine="scatter_add")
    else:
        p = synth.PRESETS[name]
    w = synth.make_weights(p, device=DEV)
    x = synth.make_x(p, w.w_router, device=DEV)
    wd = device_weights(w)
    if expert in ("e4m3", "e4m3_ue8m0"):
        wd = quantize_device_weights(wd, ue8m0=expert == "e4m3_ue8m0")
    W = B.make_weights(**wd)
    cfg = B.config_from_preset(p)
    b0 = synth.make_bias(p, device=DEV)
    gamma = 1e-3

    # eager: two steps
    ws_e = B.alloc_workspace(cfg)
    b_e = b0.clone()
    eager = []
    for _ in range(2):
        o = _buffers(p)
        _call(B, cfg, x, W, b_e, gamma, o, ws_e)
        eager.append(({k: v.clone() for k, v in o.items()}, b_e.clone()))
    torch.cuda.synchronize()
    assert B.moe_device_error(ws_e) == 0

    # graph: one eager call first (creates the library's side stream; gamma 0
    # leaves the bias alone), then capture one step and replay it twice
    ws_g = B.alloc_workspace(cfg)
    b_g = b0.clone()
    o = _buffers(p)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _call(B, cfg, x, W, b_g, 0.0, o, ws_g)
    torch.cuda.synchronize()
    assert torch.equal(b_g, b0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(B, cfg, x, W, b_g, gamma, o, ws_g)
    for step in range(2):
        o["out"].fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref, ref_bias = eager[step]
        for k in ("out", "idx", "gate", "counts", "mom"):
            if k == "out" and expert == "scatter_add":
                # the K fp32 reductions per element land in any order: equal to
                # the last bit of the bf16 output
                d = (o[k].float() - ref[k].float()).abs().max().item()
                assert d <= 2 ** -7 * ref[k].float().abs().max().item(), (step, d)
                continue
            assert torch.equal(o[k], ref[k]), (step, k)
        assert torch.equal(b_g, ref_bias), step
    assert B.moe_device_error(ws_g) == 0
