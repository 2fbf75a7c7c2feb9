"""Data-parallel replicas of the layer: the one exchange step.

Every rank holds all expert weights and routes its own batch of T tokens; the
tokens are independent, so the forward pass needs no communication. The
auxiliary-loss-free bias update, however, balances the load of the whole
step ("DeepSeek-V3技术报告" digest, mpbf.cn, section 2.2: the bias follows the
expert load of the batch): the per-expert counts of all ranks are summed
(an all-reduce of E int32, 1 KB at E = 256) and every rank applies the same
+/- gamma update with the global token count, so the replicated bias stays
identical on all ranks.
"""
from __future__ import annotations

from typing import Callable, Optional


def global_bias_update(counts, tokens_per_rank: int, update: Callable[[object, int], None],
                       group=None, dist=None) -> int:
    """Sums `counts` over the ranks of `group` in place, then calls
    update(counts, global_tokens). Returns the global token count."""
    if dist is None:
        import torch.distributed as dist
    world = dist.get_world_size(group)
    if world > 1:
        dist.all_reduce(counts, group=group)
    total = tokens_per_rank * world
    update(counts, total)
    return total


def device_bias_update(cfg, gamma: float, bias, max_over_mean=None, stream=None):
    """The `update` of global_bias_update for device tensors: moe_bias_update
    with a copy of the config whose token count is the global one."""
    from . import binding as B

    def update(counts, total_tokens: int):
        g = B.moe_config(*[getattr(cfg, f) for f, _ in B.moe_config._fields_])
        g.T = total_tokens
        B.moe_bias_update(g, counts, gamma, bias, max_over_mean, stream)

    return update
