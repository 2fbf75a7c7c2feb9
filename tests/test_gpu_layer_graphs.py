"""CUDA-graph replay of moe_layer_forward: the second call with the same
arguments is captured and later ones replay the graph. Replays must give the
same bits as launching the kernels one by one (outputs, routing, counts and
the bias trajectory), the stage events must be re-targeted at every replay,
and a new argument set must get its own graph."""
import pytest
import torch

from mixture_experts_layer_100_b300 import synth
from tests.layer_helpers import DEV, device_weights

pytestmark = pytest.mark.gpu

SHAPES = {
    # bf16, gather combine, contiguous rows
    "t515_d384_e32": dict(T=515, d=384, E=32, G=8, K=6, M=3, I=384, S=2),
    # bf16, zero-padded expert layout (T * K >= 128 E)
    "t520_d256_e8_padded": dict(T=520, d=256, E=8, G=4, K=2, M=2, I=128, S=1),
    # scatter-add combine: the fp32 accumulator and the side stream's down projection
    "t300_d256_e16_scatter": dict(T=300, d=256, E=16, G=4, K=4, M=2, I=256, S=1, combine="scatter_add"),
    # fp32 layer: tf32 pairs split at the start of every call
    "t256_d256_e16_f32": dict(T=256, d=256, E=16, G=4, K=4, M=2, I=128, S=1, dtype="f32", expert_dtype="f32"),
}


def _preset(name):
    return synth.PRESETS["mid_t4096_d2048_e64_bf16"].replace(name=name, zipf=False, bias="u0.01", **SHAPES[name])


class Layer:
    def __init__(self, p):
        from mixture_experts_layer_100_b300 import binding as B
        self.B, self.p = B, p
        w = synth.make_weights(p)
        self.wd = device_weights(w)
        self.W = B.make_weights(**self.wd)
        self.x = synth.make_x(p, w.w_router).to(DEV)
        self.b0 = synth.make_bias(p).to(DEV)
        self.cfg = B.config_from_preset(p)
        self.ws = B.alloc_workspace(self.cfg)
        dt = synth.torch_dtype(p.dtype)
        self.out = torch.empty(p.T, p.d, dtype=dt, device=DEV)
        self.idx = torch.empty(p.T, p.K, dtype=torch.int32, device=DEV)
        self.gate = torch.empty(p.T, p.K, dtype=torch.float32, device=DEV)
        self.counts = torch.empty(p.E, dtype=torch.int32, device=DEV)
        self.mom = torch.empty(1, dtype=torch.float32, device=DEV)
        self.bias = self.b0.clone()

    def step(self, x=None):
        self.B.moe_layer_forward(self.cfg, self.x if x is None else x, self.W, self.bias, self.p.gamma, self.out,
                                 self.idx, self.gate, self.counts, self.mom, self.ws)

    def run(self, n, graphs):
        self.B.moe_set_layer_graphs(graphs)
        self.bias.copy_(self.b0)
        hist = []
        try:
            for _ in range(n):
                self.step()
                hist.append([t.clone() for t in (self.out, self.idx, self.gate, self.counts, self.bias, self.mom)])
            torch.cuda.synchronize()
        finally:
            self.B.moe_set_layer_graphs(True)
        assert self.B.moe_device_error(self.ws) == 0
        return hist


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_graph_replay_gives_the_eager_bits(name):
    L = Layer(_preset(name))
    eager = L.run(5, graphs=False)
    graph = L.run(5, graphs=True)
    assert L.B.moe_layer_graphs_kept() >= 1
    scatter = SHAPES[name].get("combine") == "scatter_add"
    for step, (a, b) in enumerate(zip(eager, graph)):
        for j, (u, v) in enumerate(zip(a, b)):
            if scatter and j == 0:
                # the scatter-add combine's fp32 reductions have no fixed order,
                # so two runs of the same kernels may differ by a bf16 ulp
                uf, vf = u.float(), v.float()
                assert (uf - vf).abs().max() <= 2.0 ** -7 * uf.abs().max(), step
            else:
                assert torch.equal(u, v), (step, j)
    # the bias moved: the replays ran the update, step after step
    assert not torch.equal(graph[0][4], graph[-1][4])


def test_stage_events_are_retargeted_at_every_replay():
    L = Layer(_preset("t515_d384_e32"))
    B = L.B
    n = 6
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n)]
    for row in ev:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        t0.record()
        for i in range(n):
            B.moe_set_stage_events(ev[i])
            L.step()
        t1.record()
        torch.cuda.synchronize()
    finally:
        B.moe_set_stage_events(None)
    total = t0.elapsed_time(t1)
    spans = [ev[i][0].elapsed_time(ev[i][7]) for i in range(n)]
    # every call's events were recorded by its own launch, in order
    for i in range(n):
        parts = [ev[i][j].elapsed_time(ev[i][j + 1]) for j in range(7)]
        assert min(parts) >= 0.0 and spans[i] > 0.0
        if i:
            assert ev[i - 1][7].elapsed_time(ev[i][0]) >= 0.0
    assert sum(spans) <= total * 1.01
    assert B.moe_device_error(L.ws) == 0


def test_each_argument_set_gets_its_own_graph():
    L = Layer(_preset("t515_d384_e32"))
    x2 = torch.roll(L.x, shifts=1, dims=0).contiguous()
    outs = {}
    for graphs in (False, True):
        L.B.moe_set_layer_graphs(graphs)
        L.bias.copy_(L.b0)
        got = []
        for i in range(6):  # alternate two inputs: two argument sets, both replayed
            L.step(L.x if i % 2 == 0 else x2)
            got.append(L.out.clone())
        torch.cuda.synchronize()
        outs[graphs] = got
    L.B.moe_set_layer_graphs(True)
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a, b)
    assert not torch.equal(outs[True][0], outs[True][1])
    assert L.B.moe_device_error(L.ws) == 0
