"""Data-parallel replicas on CPU ranks (gloo, world size 2): the count
all-reduce and the global token count must give every rank the bias update
that the whole batch would get in one process."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from mixture_experts_layer_100_b300 import dp, synth
from oracle import moe_oracle as om

T, E, G, K, M, GAMMA = 96, 16, 4, 4, 2, 1e-3


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _batch(rank):
    return synth.make_scores(T, E, seed=100 + rank, kind="skewed").numpy()


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = np.zeros(E, np.float32)
        for _ in range(3):  # three steps; each rank routes only its own batch
            idx, _ = om.select_experts(_batch(rank), b, G, K, M)
            counts = torch.from_numpy(om.expert_counts(idx, E).astype(np.int32))
            state = {}

            def update(c, total):
                state["b"] = om.bias_update(c.numpy(), b, GAMMA, total, K)
                state["total"] = total

            dp.global_bias_update(counts, T, update)
            b = state["b"]
            assert state["total"] == T * world
        out[rank] = torch.from_numpy(b)
    finally:
        dist.destroy_process_group()


def test_two_rank_bias_update_matches_one_process():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # one process over the concatenated batch
    b = np.zeros(E, np.float32)
    for _ in range(3):
        idx = np.concatenate([om.select_experts(_batch(r), b, G, K, M)[0] for r in range(world)])
        b = om.bias_update(om.expert_counts(idx, E), b, GAMMA, T * world, K)
    np.testing.assert_array_equal(out[0].numpy(), b)
    np.testing.assert_array_equal(out[1].numpy(), b)
