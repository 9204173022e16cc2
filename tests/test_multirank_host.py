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


def test_threaded_oracle_timing_writes_the_single_threaded_bytes():
    # the all-cores CPU baseline runs the unchanged oracle on slices of the
    # outputs in several threads at once; the slices write disjoint slots, so
    # the cache must come out byte for byte as one single-threaded call leaves it
    import sys

    import numpy as np

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import bench
    import oracle
    from kv_cache_compression_c128_gb300 import inputs

    case = inputs.make_case(2, 2048, 64, seed=inputs.BASE_SEED + 6000, kv_fill=9)
    kvs = []
    _, n = bench.time_oracle_threads(case, 5, min_seconds=1e9, max_passes=2, kv_out=kvs)
    assert n == 2 * case.num_outputs and len(kvs) == 1
    kv1 = case.kv_cache.copy()
    res = oracle.compress(case.state_bits, case.token_to_req, case.positions,
                          case.boundary_token_indices, case.block_table, case.rms_norm_weight,
                          case.cos_sin_cache, case.kv_slot_mapping, kv1, case.block_size,
                          case.compress_ratio, case.rms_norm_eps)
    assert res["status"] == 0
    assert np.array_equal(kvs[0], kv1)
    assert not np.array_equal(kv1, case.kv_cache)
