"""Host logic of bench.py's multi-rank path, on two gloo ranks (CPU only).

The compressor's outputs are independent, so under torchrun every rank
compresses its own batch (weak scaling) and the only cross-rank step is the
timing reduction: the maximum elapsed time over ranks.  These tests run that
reduction, the per-rank seeding and the environment parsing in two real
processes joined by a gloo process group on 127.0.0.1.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.dist_env()
        elapsed = 0.25 * (rank + 1)              # rank 1 is the slower one
        t_max = bench.max_over_ranks(elapsed)
        bench.barrier()
        out.put((rank, env, t_max, bench.rank_seed(20260614, rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_distinct_seeds():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, env0, t0, s0), (r1, env1, t1, s1) = res
    assert env0 == (0, 2, 0) and env1 == (1, 2, 1)
    assert t0 == t1 == pytest.approx(0.5)       # both ranks see the max
    assert s0 != s1                             # independent batches per rank


def test_single_process_reduction_is_identity():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.rank_seed(7, 0) == 7
