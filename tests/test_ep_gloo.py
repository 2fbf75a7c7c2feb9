"""Expert parallelism on CPU ranks (gloo; the row reorders are plain torch
indexing here, the library's kernels on GPUs): each rank routes its own tokens,
sends its permuted rows to the ranks that hold their experts, runs its local
experts on what it receives, and gets its rows' outputs back; combined with
the gates, every rank's layer output must equal the single-process oracle's
("DeepSeek-V3技术报告" digest, mpbf.cn, section 3.3). The plans are also
checked against a brute-force construction, and the group limit must bound
the ranks one token reaches when each rank holds one group."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixture_experts_layer_100_b300 import ep
from oracle import moe_oracle as om

E, G, K, M, D, I, S = 16, 4, 4, 2, 64, 32, 1


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _weights():
    rng = np.random.default_rng(0)
    return {"w_router": rng.standard_normal((E, D)) * 0.2, "w13": rng.standard_normal((E, 2 * I, D)) * 0.1,
            "w2": rng.standard_normal((E, D, I)) * 0.1, "ws13": rng.standard_normal((S, 2 * I, D)) * 0.1,
            "ws2": rng.standard_normal((S, D, I)) * 0.1}


def _tokens(rank):
    return np.random.default_rng(100 + rank).standard_normal((40 + 7 * rank, D))


def _scatter_rows(src, idx, n_dst):
    dst = src.new_empty((n_dst,) + tuple(src.shape[1:]))
    dst[idx] = src
    return dst


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = _weights()
        x = _tokens(rank)
        b = np.zeros(E, np.float32)
        s = om.router_scores(x, w["w_router"])
        idx, gate = om.select_experts(s, b, G, K, M)
        counts = om.expert_counts(idx, E)
        offsets = om.exclusive_offsets(counts)
        st, sp = om.permutation(idx, E)
        xp = torch.from_numpy(x[st])
        rows, local_off, plan = ep.dispatch(xp, torch.from_numpy(offsets), torch.from_numpy(counts), world,
                                            gather_rows=lambda src, idx: src[idx])
        per = E // world
        y_local = torch.empty_like(rows)
        lo = local_off.numpy()
        for el in range(per):
            e = rank * per + el
            if lo[el + 1] > lo[el]:
                y_local[lo[el]:lo[el + 1]] = torch.from_numpy(
                    om.swiglu_ffn(rows[lo[el]:lo[el + 1]].numpy(), w["w13"][e], w["w2"][e]))
        yp = ep.combine_back(y_local, plan, scatter_rows=_scatter_rows).numpy()
        res = om.shared_output(x, w["ws13"], w["ws2"])
        for k in range(K):
            res += gate[:, k:k + 1].astype(np.float64) * yp[sp[:, k]]
        ref = om.layer_forward(x, w["w_router"], w["w13"], w["w2"], w["ws13"], w["ws2"], b, G, K, M)["out"]
        reached = ep.ranks_reached(torch.from_numpy(idx), E, world)
        out[rank] = (float(np.abs(res - ref).max() / np.abs(ref).max()), int(reached.max()),
                     int(plan["recv_splits"].sum()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_expert_parallel_layer_matches_single_process(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    total_rows = sum(out[r][2] for r in range(world))
    assert total_rows == sum(_tokens(r).shape[0] for r in range(world)) * K  # every (token, slot) row once
    for r in range(world):
        err, reached, _ = out[r]
        assert err <= 1e-12, (r, err)
        if world == G:  # one group per rank: the group limit bounds the ranks reached
            assert reached <= M


def test_recv_plan_against_brute_force():
    rng = np.random.default_rng(3)
    R, El = 3, 4
    cm = rng.integers(0, 5, (R, El))
    # receive buffer: source-major, expert-major inside a source; label every row
    labels = [(s, e, j) for s in range(R) for e in range(El) for j in range(cm[s, e])]
    recv_splits, local_off, gather = ep.recv_plan(torch.from_numpy(cm))
    assert recv_splits.tolist() == cm.sum(1).tolist()
    want = [(s, e, j) for e in range(El) for s in range(R) for j in range(cm[s, e])]
    assert [labels[g] for g in gather.tolist()] == want
    assert local_off.tolist() == [0] + np.cumsum(cm.sum(0)).tolist()


def test_send_splits_follow_the_expert_offsets():
    counts = torch.tensor([3, 0, 2, 5, 1, 1, 0, 4])
    off = torch.zeros(9, dtype=torch.int64)
    off[1:] = torch.cumsum(counts, 0)
    assert ep.send_splits(off, 4).tolist() == [3, 7, 2, 4]
    assert ep.send_splits(off, 2).tolist() == [10, 6]
    assert ep.send_expert_counts(counts, 4).tolist() == [[3, 0], [2, 5], [1, 1], [0, 4]]
    with pytest.raises(ValueError):
        ep.send_splits(off, 3)
