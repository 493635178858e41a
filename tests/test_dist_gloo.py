"""The multi-replica host path on CPU: two gloo ranks sum their parameter
gradients with one all-reduce and agree on the job's step time (max)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from selective_state_space_114_b300 import dist as sdist
        g = {"dA": torch.full((4, 16), float(rank + 1)), "dD": torch.arange(4.0) * (rank + 1),
             "ddelta_bias": None, "du": torch.full((2, 4, 8), float(rank))}
        sdist.allreduce_param_grads(g)
        t = sdist.max_over_ranks(1.5 + rank)
        q.put((rank, g["dA"].clone(), g["dD"].clone(), g["du"].clone(), t,
               sdist.rank_seed(1001, rank)))
    finally:
        dist.destroy_process_group()


def test_two_rank_param_grad_allreduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, dA, dD, du, t, seed in res:
        assert torch.all(dA == 3.0)                      # 1 + 2
        assert torch.equal(dD, torch.arange(4.0) * 3)    # summed
        assert torch.all(du == float(rank))              # per-row outputs untouched
        assert t == 2.5                                  # max over ranks
    assert res[0][5] != res[1][5]                        # distinct data per replica
