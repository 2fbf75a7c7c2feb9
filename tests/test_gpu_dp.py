"""The data-parallel bias update as bench.py runs it with more than one rank:
dp.global_bias_update with dp.device_bias_update, i.e. moe_bias_update on the
device with the global token count, after the count exchange. The exchange
is a stand-in here (one GPU): it adds a second rank's counts and reports a
world of two, so the update must use the summed counts and twice the local
token count ("DeepSeek-V3技术报告" digest, mpbf.cn, section 2.2: the bias
follows the load of the whole batch)."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_100_b300 import dp, synth
from oracle import cpp
from tests.layer_helpers import DEV, device_weights, run_layer

pytestmark = pytest.mark.gpu


class TwoRankExchange:
    """torch.distributed stand-in: world size 2, the other rank's counts
    given up front."""

    def __init__(self, other):
        self.other = other
        self.calls = 0

    def get_world_size(self, group=None):
        return 2

    def all_reduce(self, t, group=None):
        self.calls += 1
        t.add_(self.other)


def test_device_bias_update_uses_the_global_batch():
    from mixture_experts_layer_100_b300 import binding as B
    p = synth.PRESETS["mid_t4096_d2048_e64_bf16"].replace(T=700, d=256, I=128, E=64, G=8, K=6, M=3, S=1)
    w = synth.make_weights(p)
    x = synth.make_x(p, w.w_router).to(DEV)
    b0 = synth.make_bias(p)
    bias = b0.clone().to(DEV)
    res = run_layer(p, device_weights(w), x, bias, gamma=0.0)  # the layer without its own update
    counts = res["counts"]
    local = counts.cpu().numpy().astype(np.int32)
    # the second rank's load: the same total T*K, spread differently
    other = np.roll(local, 5) + np.where(np.arange(p.E) % 2 == 0, 3, -3).astype(np.int32)
    other[other < 0] = 0
    other[0] += p.T * p.K - other.sum()
    ex = TwoRankExchange(torch.from_numpy(other).to(DEV))
    cfg = B.config_from_preset(p)
    mom = torch.empty(1, dtype=torch.float32, device=DEV)
    total = dp.global_bias_update(counts, p.T, dp.device_bias_update(cfg, p.gamma, bias, mom), dist=ex)
    torch.cuda.synchronize()
    assert ex.calls == 1 and total == 2 * p.T
    both = local + other
    want = cpp.bias_update(both, b0.numpy(), p.gamma, 2 * p.T, p.K)
    np.testing.assert_array_equal(bias.cpu().numpy(), want)
    assert mom.item() == cpp.load_max_over_mean(both, 2 * p.T, p.K)
    # with the local token count the update would differ: the test can tell
    assert not np.array_equal(want, cpp.bias_update(both, b0.numpy(), p.gamma, p.T, p.K))
