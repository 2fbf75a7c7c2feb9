"""Expert-parallel dispatch and combine with R ranks emulated on one GPU
("DeepSeek-V3技术报告" digest, mpbf.cn, section 3.3). Rank r holds experts
[r E/R, (r+1) E/R). The exchange between ranks is emulated by slicing and
concatenating device buffers (what the all-to-all does); every other step
runs in the library's kernels: routing and permutation on each rank's own
tokens, the receive-side reorder (moe_gather_rows), the rank's grouped expert
GEMMs on its E/R experts, the inverse reorder (moe_scatter_rows), and the
combine on the rank that owns the tokens. Every row of the expert GEMMs is
computed by the same instructions whichever rows share its tile, so each
rank's output must equal the single-GPU layer's bit for bit."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_100_b300 import ep, synth
from tests.layer_helpers import DEV, device_weights, run_layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 4])
def test_emulated_expert_parallel_layer_is_the_single_gpu_layer(world):
    from mixture_experts_layer_100_b300 import binding as B
    base = synth.PRESETS["mid_t4096_d2048_e64_bf16"].replace(d=256, I=128, E=32, G=4, K=4, M=2, S=1, zipf=False)
    El = base.E // world
    w = synth.make_weights(base)
    wd = device_weights(w)
    W = B.make_weights(**wd)
    ranks = []
    for r in range(world):
        p = base.replace(T=300 + 57 * r, seed=r + 1)
        x = synth.make_x(p, w.w_router).to(DEV)
        b = synth.make_bias(p).to(DEV)
        ref = run_layer(p, wd, x, b)  # the single-GPU layer on this rank's tokens
        cfg = B.config_from_preset(p)
        ws = B.alloc_workspace(cfg)
        T, K, E, d = p.T, p.K, p.E, p.d
        idx = torch.empty(T, K, dtype=torch.int32, device=DEV)
        gate = torch.empty(T, K, dtype=torch.float32, device=DEV)
        counts = torch.empty(E, dtype=torch.int32, device=DEV)
        off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
        st = torch.empty(T * K, dtype=torch.int32, device=DEV)
        sp = torch.empty(T, K, dtype=torch.int32, device=DEV)
        xp = torch.empty(T * K, d, dtype=torch.bfloat16, device=DEV)
        B.moe_route(cfg, x, wd["w_router"], None, b, None, idx, gate, counts, ws)
        B.moe_permute(cfg, idx, counts, off, st, sp, x, xp, None, ws)
        ranks.append(dict(p=p, x=x, ref=ref, cfg=cfg, ws=ws, gate=gate, counts=counts, off=off, sp=sp, xp=xp,
                          ss=ep.send_splits(off, world).cpu()))
    torch.cuda.synchronize()

    # dispatch: rank q receives from every source s the slice of s's rows for q's experts
    ws_ep = B.alloc_workspace(ranks[0]["cfg"])
    gather_rows, scatter_rows = ep.device_row_moves(ws_ep)
    back = [[None] * world for _ in range(world)]  # back[s][q]: q's outputs for s's rows
    for q in range(world):
        parts, cm = [], []
        for s in range(world):
            o = ranks[s]["off"].cpu().numpy()
            parts.append(ranks[s]["xp"][o[q * El]:o[(q + 1) * El]])
            cm.append(ranks[s]["counts"].view(world, El)[q])
        recv = torch.cat(parts)
        recv_splits, local_off, gather = ep.recv_plan(torch.stack(cm).cpu())
        assert recv_splits.tolist() == [x.shape[0] for x in parts]
        rows = gather_rows(recv, gather.to(DEV))
        n = rows.shape[0]
        # the rank's grouped expert GEMMs on its E/R experts
        cfg_q = B.make_config(n, base.d, El, 1, 1, 1, base.I, 0, 1, act="bf16")
        ws_q = B.alloc_workspace(cfg_q)
        Wq = B.make_weights(w13=wd["w13"][q * El:(q + 1) * El].contiguous(),
                            w2=wd["w2"][q * El:(q + 1) * El].contiguous())
        y = torch.empty_like(rows)
        B.moe_grouped_ffn(cfg_q, rows, None, local_off.to(torch.int32).to(DEV), Wq, y, ws_q)
        y_recv = scatter_rows(y, gather.to(DEV), n)
        starts = np.concatenate([[0], np.cumsum(recv_splits.numpy())])
        for s in range(world):
            back[s][q] = y_recv[starts[s]:starts[s + 1]]
        torch.cuda.synchronize()
        assert B.moe_device_error(ws_q) == 0

    # combine on the rank that owns the tokens: its rows come back in its own expert-major order
    for s, rk in enumerate(ranks):
        yp = torch.cat(back[s])
        assert yp.shape[0] == rk["p"].T * rk["p"].K
        out = torch.empty_like(rk["ref"]["out"])
        B.moe_combine(rk["cfg"], yp, rk["sp"], rk["gate"], rk["x"], W, out, rk["ws"])
        torch.cuda.synchronize()
        assert B.moe_device_error(rk["ws"]) == 0
        assert torch.equal(out, rk["ref"]["out"]), s
    assert B.moe_device_error(ws_ep) == 0


def test_row_moves_round_trip_and_bad_index():
    from mixture_experts_layer_100_b300 import binding as B
    cfg = B.make_config(8, 128, 16, 4, 4, 2, 128, 1, 2, act="bf16")
    ws = B.alloc_workspace(cfg)
    src = torch.randn(100, 72, device=DEV)  # 288-byte rows: 16-byte vectors
    perm = torch.randperm(100, device=DEV).to(torch.int32)
    g = torch.empty_like(src)
    B.moe_gather_rows(src, perm, g, ws)
    assert torch.equal(g, src[perm.long()])
    back = torch.zeros_like(src)
    B.moe_scatter_rows(g, perm, back, ws)
    assert torch.equal(back, src)
    odd = torch.randn(50, 3, device=DEV)  # 12-byte rows: 4-byte words
    idx = torch.arange(49, -1, -1, device=DEV, dtype=torch.int32)
    o = torch.empty_like(odd)
    B.moe_gather_rows(odd, idx, o, ws)
    assert torch.equal(o, odd.flip(0))
    torch.cuda.synchronize()
    assert B.moe_device_error(ws) == 0
    bad = perm.clone()
    bad[7] = 100  # one past the end: skipped and reported
    B.moe_gather_rows(src, bad, g, ws)
    assert B.moe_device_error(ws) == 0x203
