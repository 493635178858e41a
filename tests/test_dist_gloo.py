"""The multi-replica host path on CPU: two gloo ranks sum their parameter
gradients with one all-reduce and agree on the job's step time (max)."""
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, store_path, q):
    # file rendezvous: no TCP port to race for
    dist.init_process_group("gloo", init_method=f"file://{store_path}", rank=rank,
                            world_size=world)
    try:
        from selective_state_space_114_b300 import dist as sdist
        g = {"dA": torch.full((4, 16), float(rank + 1)), "dD": torch.arange(4.0) * (rank + 1),
             "ddelta_bias": None, "du": torch.full((2, 4, 8), float(rank))}
        sdist.allreduce_param_grads(g)
        t = sdist.max_over_ranks(1.5 + rank)
        # numpy copies travel by value (torch tensors would be shared by file
        # descriptor, which dies with this process)
        q.put((rank, g["dA"].numpy().copy(), g["dD"].numpy().copy(), g["du"].numpy().copy(),
               t, sdist.rank_seed(1001, rank)))
    finally:
        dist.destroy_process_group()


def test_two_rank_param_grad_allreduce(tmp_path):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    store = str(tmp_path / "rendezvous")
    procs = [ctx.Process(target=_worker, args=(r, 2, store, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(2)), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, dA, dD, du, t, seed in res:
        assert (dA == 3.0).all()                              # 1 + 2
        assert (dD == torch.arange(4.0).numpy() * 3).all()    # summed
        assert (du == float(rank)).all()                      # per-row outputs untouched
        assert t == 2.5                                  # max over ranks
    assert res[0][5] != res[1][5]                        # distinct data per replica
