"""The multi-process (N > 1) host logic of bench.py, on CPU with the gloo backend.

The selection path partitions by query with no exchange step: N ranks each run
their own calls (weak scaling) and the job is timed by its slowest rank.  These
tests run two gloo ranks and check the max-over-ranks reduction, the whole-job
figure, and that selecting query shards independently gives the same ids as
selecting all queries at once (so no collective is needed on the data path).
The KV-sharded form (each rank holds a range of every query's blocks) has one
exchange, an all-gather of the ranks' candidates; its host flow runs here on
two and three gloo ranks with the oracle standing in for the library's stages.
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
        from workloads import inputs
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
    from workloads import inputs
    sc = inputs.normal_scores(42, 8, 300).astype(np.float64)
    nb = np.array([300, 299, 120, 40, 3, 300, 255, 1], dtype=np.int32)
    want = oracle.select(sc, nb, 16).tolist()
    for rank in range(world):
        mx, ids = out[rank]
        assert mx == 2.5
        assert ids == want


def _stage_a_oracle(scores, n_blocks, k, cand_scores, cand_ids, ws, offset, max_blocks, active):
    """Stage A as the library defines it, computed by the oracle: the shard's selection
    (local ids ascending, -1 padded) moved to global ids, with each candidate's score."""
    import oracle
    s = scores.numpy()
    loc = oracle.select_f32(s, n_blocks.numpy(), k)
    rows = np.arange(s.shape[0])[:, None]
    cand_ids.copy_(torch.from_numpy(np.where(loc >= 0, loc + offset, -1).astype(np.int32)))
    cand_scores.copy_(torch.from_numpy(np.where(loc >= 0, s[rows, np.maximum(loc, 0)], -np.inf).astype(np.float32)))


def _stage_b_reference(all_scores, all_ids, ids):
    """Stage B written out: per query, the k first of every shard's candidates in
    (score descending, global id ascending), ids ascending, -1 padded."""
    G, nq, k = all_ids.shape
    for q in range(nq):
        sc = all_scores[:, q, :].reshape(-1).numpy().astype(np.float64)
        i = all_ids[:, q, :].reshape(-1).numpy()
        keep = i >= 0
        sc, i = sc[keep], i[keep]
        order = np.lexsort((i, -sc))
        out = np.full(k, -1, dtype=np.int32)
        sel = np.sort(i[order[:k]])
        out[:len(sel)] = sel
        ids[q] = torch.from_numpy(out)


def _sharded_worker(rank, world, port, bounds, kind, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    try:
        from sparse_attention_kv_gb300 import sharded
        from workloads import inputs
        sc, nb, k = _sharded_case(kind)
        lo, hi = bounds[rank], bounds[rank + 1]
        local = torch.from_numpy(np.ascontiguousarray(sc[:, lo:hi]))
        n_loc = torch.from_numpy(np.clip(nb - lo, 0, hi - lo).astype(np.int32))
        ids = torch.full((sc.shape[0], k), -7, dtype=torch.int32)
        sharded.select_kv_sharded(local, n_loc, k, lo, ids, max_blocks=hi - lo, stage_a=_stage_a_oracle,
                                  stage_b=_stage_b_reference)
        out[rank] = ids.numpy().tolist()
    finally:
        dist.destroy_process_group()


def _sharded_case(kind):
    from workloads import inputs
    if kind == "normal":
        sc = inputs.normal_scores(4242, 12, 500)
    else:
        sc = inputs.level_scores(4243, 12, 500)   # many ties, across the shard boundary too
    nb = np.array([500, 499, 260, 250, 249, 3, 0, 1, 500, 131, 400, 17], dtype=np.int32)
    return sc, nb, 16


@pytest.mark.parametrize("kind", ["normal", "levels"])
@pytest.mark.parametrize("world,bounds", [(2, [0, 250, 500]), (3, [0, 131, 399, 500])])
def test_kv_sharded_select_over_gloo_ranks(kind, world, bounds):
    """Each rank holds a range of every query's blocks; candidates all-gathered into
    [world, nq, k] and merged give, on every rank, the unsharded selection."""
    import oracle
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_sharded_worker, args=(world, port, bounds, kind, out), nprocs=world, join=True)
    sc, nb, k = _sharded_case(kind)
    want = oracle.select_f32(sc, nb, k)
    for rank in range(world):
        np.testing.assert_array_equal(np.array(out[rank]), want)


def test_job_figure_divides_by_ranks():
    import bench
    assert bench.job_us_per_call(0.040, 1) == pytest.approx(40.0)
    assert bench.job_us_per_call(0.040, 4) == pytest.approx(10.0)
    assert bench.max_over_ranks(3.0) == 3.0   # no process group: identity
