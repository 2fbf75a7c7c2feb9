"""Expert parallelism across ranks: the index plans of the all-to-all
dispatch and combine ("DeepSeek-V3技术报告" digest, mpbf.cn, section 3.3:
tokens are sent to the nodes that hold their experts and the expert outputs
are sent back and combined; node-limited routing bounds how many nodes one
token reaches).

Placement: rank r of R holds the experts [r * E/R, (r+1) * E/R). With one
expert group per rank (G = R), the group limit M of the routing bounds the
ranks one token's rows go to by M.

Dispatch. moe_permute orders a rank's (token, slot) rows expert-major; with
contiguous placement that order is also destination-major, so the permuted
rows xp are the send buffer as they are: rank r receives the slice
[offsets[r E/R], offsets[(r+1) E/R]). Beside the rows, each rank sends every
destination the per-expert counts of its slice (E/R integers), so that the
receiver knows how its buffer, which arrives source-major, splits by expert.

Local experts. recv_plan turns the [R sources, E/R local experts] count
matrix into the receive splits, the local expert offsets and a gather index
that reorders the received rows expert-major (for each local expert, the
rows of source 0, then source 1, ...); the grouped expert GEMMs run on that
order.

Combine. The outputs go back through the inverse of that gather, the reverse
all-to-all returns every row to the rank and position it came from, which is
the single-GPU routed output yp in expert-major order; the gate-weighted
combine then runs unchanged (moe_combine).

Only index arithmetic lives here (torch integer ops, host or device); the
exchange is torch.distributed's all_to_all_single, and the row reorders are
the library's moe_gather_rows / moe_scatter_rows kernels on the device
(device_row_moves), or whatever row-move functions the caller passes.
"""
from __future__ import annotations

from typing import Tuple

import torch


def experts_per_rank(E: int, world: int) -> int:
    if world <= 0 or E % world != 0:
        raise ValueError(f"{E} experts do not split evenly over {world} ranks")
    return E // world


def _exclusive_cumsum(v: torch.Tensor, dim: int = 0) -> torch.Tensor:
    return torch.cumsum(v, dim=dim) - v


def send_splits(offsets: torch.Tensor, world: int) -> torch.Tensor:
    """Rows this rank sends to each rank: the per-rank slices of the expert
    offsets [E + 1] that moe_permute writes. Returns int64 [world]."""
    E = offsets.numel() - 1
    per = experts_per_rank(E, world)
    o = offsets.to(torch.int64)[torch.arange(0, world + 1, device=offsets.device) * per]
    return o[1:] - o[:-1]


def send_expert_counts(counts: torch.Tensor, world: int) -> torch.Tensor:
    """Per-destination expert counts [world, E/R] (row r: this rank's rows for
    each of rank r's experts), exchanged with one all-to-all of E integers."""
    E = counts.numel()
    return counts.to(torch.int64).view(world, experts_per_rank(E, world))


def recv_plan(count_matrix: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """From count_matrix [R sources, El local experts] (source s sends
    count_matrix[s, e] rows for local expert e, expert-major within the
    source) build:
      recv_splits [R]     rows received from each source;
      local_offsets [El + 1] expert offsets of the expert-major local order;
      gather [N]          receive-buffer position of each row of the local
                          order (local order: for e, for s, the rows in the
                          order they arrived).
    """
    cm = count_matrix.to(torch.int64)
    R, El = cm.shape
    dev = cm.device
    recv_splits = cm.sum(1)
    src_base = _exclusive_cumsum(recv_splits)                  # first position of source s
    within = _exclusive_cumsum(cm, dim=1)                      # start of expert e inside source s
    local_counts = cm.sum(0)
    local_offsets = torch.zeros(El + 1, dtype=torch.int64, device=dev)
    local_offsets[1:] = torch.cumsum(local_counts, 0)
    # blocks in local order: (e, s) for e ascending, s ascending
    blk_len = cm.t().reshape(-1)                               # [El * R]
    blk_src = (src_base[None, :] + within.t()).reshape(-1)     # receive start of each block
    n = int(blk_len.sum())
    blk_local_start = _exclusive_cumsum(blk_len)
    blk_id = torch.repeat_interleave(torch.arange(El * R, device=dev), blk_len)
    j = torch.arange(n, device=dev) - blk_local_start[blk_id]
    gather = blk_src[blk_id] + j
    return recv_splits, local_offsets, gather


def ranks_reached(topk_idx: torch.Tensor, E: int, world: int) -> torch.Tensor:
    """Distinct destination ranks of each token's rows [T] (at most M when the
    E/R experts of a rank form one routing group and at most M groups are
    chosen): the row count a per-rank de-duplicated dispatch would send."""
    per = experts_per_rank(E, world)
    dest = topk_idx.to(torch.int64) // per
    onehot = torch.zeros(topk_idx.shape[0], world, dtype=torch.bool, device=topk_idx.device)
    onehot.scatter_(1, dest, True)
    return onehot.sum(1)


def dispatch(xp: torch.Tensor, offsets: torch.Tensor, counts: torch.Tensor, world: int, gather_rows,
             group=None, dist=None):
    """All-to-all dispatch of a rank's permuted rows. gather_rows(src, idx)
    returns src's rows in idx order (on the GPU: moe_gather_rows, see
    device_row_moves). Returns (rows in local expert-major order,
    local_offsets, plan) where plan carries what combine_back needs to send
    the outputs back."""
    if dist is None:
        import torch.distributed as dist
    ss = send_splits(offsets, world)
    cm_out = send_expert_counts(counts, world).contiguous()
    cm_in = torch.empty_like(cm_out)
    dist.all_to_all_single(cm_in, cm_out, group=group)
    recv_splits, local_offsets, gather = recv_plan(cm_in)
    recv = xp.new_empty((int(recv_splits.sum()),) + tuple(xp.shape[1:]))
    dist.all_to_all_single(recv, xp[: int(ss.sum())].contiguous(), output_split_sizes=recv_splits.tolist(),
                           input_split_sizes=ss.tolist(), group=group)
    return gather_rows(recv, gather), local_offsets, {"send_splits": ss, "recv_splits": recv_splits,
                                                      "gather": gather}


def combine_back(y_local: torch.Tensor, plan, scatter_rows, group=None, dist=None) -> torch.Tensor:
    """Returns the expert outputs of this rank's own rows, in its
    expert-major order (the yp of the single-GPU layer). scatter_rows(src,
    idx, n_dst) returns dst with dst[idx[i]] = src[i]."""
    if dist is None:
        import torch.distributed as dist
    y_recv = scatter_rows(y_local, plan["gather"], y_local.shape[0])
    out = y_local.new_empty((int(plan["send_splits"].sum()),) + tuple(y_local.shape[1:]))
    dist.all_to_all_single(out, y_recv, output_split_sizes=plan["send_splits"].tolist(),
                           input_split_sizes=plan["recv_splits"].tolist(), group=group)
    return out


def device_row_moves(ws):
    """(gather_rows, scatter_rows) for device tensors, run by the library's
    moe_gather_rows / moe_scatter_rows kernels; ws is a workspace whose error
    word they report bad indices in."""
    from . import binding as B

    def gather_rows(src, idx):
        idx32 = idx.to(torch.int32).contiguous()
        dst = src.new_empty((idx32.numel(),) + tuple(src.shape[1:]))
        B.moe_gather_rows(src.contiguous(), idx32, dst, ws)
        return dst

    def scatter_rows(src, idx, n_dst):
        idx32 = idx.to(torch.int32).contiguous()
        dst = src.new_empty((n_dst,) + tuple(src.shape[1:]))
        B.moe_scatter_rows(src.contiguous(), idx32, dst, ws)
        return dst

    return gather_rows, scatter_rows
