"""The multi-process (N > 1) host logic of bench.py, on CPU with the gloo backend.

The selection path partitions by query with no exchange step: N ranks each run
their own calls (weak scaling) and the job is timed by its slowest rank.  These
tests run two gloo ranks and check the max-over-ranks reduction, the whole-job
figure, and that selecting query shards independently gives the same ids as
selecting all queries at once (so no collective is needed on the data path).
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from sparse_attention_kv_gb300 import inputs
        mx = bench.max_over_ranks(1.5 + rank)
        # this rank's shard of queries, selected on its own
        sc = inputs.normal_scores(42, 8, 300).astype(np.float64)
        nb = np.array([300, 299, 120, 40, 3, 300, 255, 1], dtype=np.int32)
        lo, hi = rank * 8 // world, (rank + 1) * 8 // world
        ids = oracle.select(sc[lo:hi], nb[lo:hi], 16)
        gathered = [None] * world
        dist.all_gather_object(gathered, ids.tolist())
        out[rank] = (mx, [row for part in gathered for row in part])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_query_shards():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    import oracle
    from sparse_attention_kv_gb300 import inputs
    sc = inputs.normal_scores(42, 8, 300).astype(np.float64)
    nb = np.array([300, 299, 120, 40, 3, 300, 255, 1], dtype=np.int32)
    want = oracle.select(sc, nb, 16).tolist()
    for rank in range(world):
        mx, ids = out[rank]
        assert mx == 2.5
        assert ids == want


def test_job_figure_divides_by_ranks():
    import bench
    assert bench.job_us_per_call(0.040, 1) == pytest.approx(40.0)
    assert bench.job_us_per_call(0.040, 4) == pytest.approx(10.0)
    assert bench.max_over_ranks(3.0) == 3.0   # no process group: identity
