"""KV-sharded selection on one GPU: qsa_block_candidates per shard, then
qsa_merge_candidates over every shard's candidates.

The blocks of each query are split into G ranges, as G GPUs would hold them; each
range's candidates are computed over a view of the score rows with its global
block offset, laid out shard-major ([G][nq][k], what an all-gather of the shards'
[nq][k] arrays leaves), and merged.  The ids must equal one selection over all
blocks (qsa_block_topk / qsa_select) and the oracle's selection over the same
scores, bit for bit: a query's selection restricted to a shard is a prefix of
that shard's order, so no selected block is lost (Strata PR #3987, "Approach").
"""
import numpy as np
import pytest

import oracle
from workloads import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from sparse_attention_kv_gb300 import qsa  # noqa: E402
from tests import parity  # noqa: E402


def sharded_ids(scores, n_blocks, k, bounds, path=qsa.PATH_AUTO):
    """ids [nq, k] of the sharded selection: shard g holds blocks [bounds[g], bounds[g + 1])."""
    nq = scores.shape[0]
    G = len(bounds) - 1
    n = n_blocks.cpu().numpy()
    cs = torch.full((G, nq, k), float("nan"), dtype=torch.float32, device="cuda")
    ci = torch.full((G, nq, k), -9, dtype=torch.int32, device="cuda")
    ws = qsa.alloc_workspace(nq, max(bounds[g + 1] - bounds[g] for g in range(G)), k)
    for g in range(G):
        lo, hi = bounds[g], bounds[g + 1]
        n_loc = torch.from_numpy(np.clip(n - lo, 0, hi - lo).astype(np.int32)).cuda()
        qsa.block_candidates(scores[:, lo:hi], n_loc, k, cs[g], ci[g], ws, block_offset=lo, max_blocks=hi - lo,
                             path=path)
    assert qsa.read_flags(ws) & qsa.ERROR_FLAGS == 0
    ids = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
    qsa.merge_candidates(cs, ci, ids)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), cs.cpu().numpy(), ci.cpu().numpy()


def whole_ids(scores, n_blocks, k):
    nq, C = scores.shape
    ids = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
    ws = qsa.alloc_workspace(nq, C, k)
    qsa.block_topk(scores, n_blocks, k, ids, ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy()


def split_points(rng, C, G, aligned):
    if G == 1:
        return [0, C]
    cuts = np.sort(rng.choice(np.arange(1, C), size=G - 1, replace=False))
    if aligned:
        cuts = np.unique(cuts // 128 * 128)
        cuts = cuts[(cuts > 0) & (cuts < C)]
    return [0, *cuts.tolist(), C]


@pytest.fixture(scope="module")
def deep_scores():
    """The deep prompt's own scores (256 queries x 8,125 blocks) and its select ids."""
    case = inputs.deep_case(2)
    q, w, kb, nb = parity.to_device(case, "cuda")
    sc = torch.empty((case.nq, case.max_blocks), dtype=torch.float32, device="cuda")
    ids = torch.empty((case.nq, case.k), dtype=torch.int32, device="cuda")
    ws = qsa.alloc_workspace(case.nq, case.max_blocks, case.k)
    qsa.select(q, w, kb, nb, case.k, ids, ws, scores=sc, active_blocks=case.active_blocks)
    torch.cuda.synchronize()
    return sc, nb, case.k, ids.cpu().numpy()


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("aligned", [True, False])
def test_deep_prompt_sharded_equals_one_select_and_oracle(deep_scores, G, aligned):
    sc, nb, k, select_ids = deep_scores
    rng = np.random.default_rng(7700 + G + 10 * aligned)
    bounds = split_points(rng, 8125, G, aligned)
    got, cs, ci = sharded_ids(sc[:, :8125], nb, k, bounds)
    np.testing.assert_array_equal(got, select_ids)
    s_np = sc.cpu().numpy()[:, :8125]
    np.testing.assert_array_equal(got, oracle.select_f32(s_np, nb.cpu().numpy(), k))
    # every candidate carries its own block's score and a global id inside its shard
    for g in range(len(bounds) - 1):
        v = ci[g] >= 0
        assert ((ci[g][v] >= bounds[g]) & (ci[g][v] < bounds[g + 1])).all()
        rows = np.nonzero(v)[0]
        np.testing.assert_array_equal(cs[g][v], s_np[rows, ci[g][v]])


@pytest.mark.parametrize("kind", ["normal", "levels", "equal"])
@pytest.mark.parametrize("k", [1, 7, 32, 64])
def test_sharded_ties_ragged_and_short_rows(kind, k):
    """Ties across shards go to the lowest global id; ragged contexts leave some
    shards without blocks; rows shorter than k give -1 padding."""
    nq, C = 40, 3000
    seed = 7800 + k
    if kind == "normal":
        sc = inputs.normal_scores(seed, nq, C)
    elif kind == "levels":
        sc = inputs.level_scores(seed, nq, C)
    else:
        sc = np.full((nq, C), 0.5, dtype=np.float32)
    rng = np.random.default_rng(seed)
    n = rng.integers(0, C + 1, size=nq).astype(np.int32)
    n[:4] = [0, 1, k - 1 if k > 1 else 0, k]
    scores = torch.from_numpy(sc).cuda()
    n_dev = torch.from_numpy(n).cuda()
    want = oracle.select_f32(sc, n, k)
    for G in (2, 3, 8):
        bounds = split_points(rng, C, G, aligned=False)
        got, _, _ = sharded_ids(scores, n_dev, k, bounds)
        np.testing.assert_array_equal(got, want, err_msg=f"G={G} bounds={bounds}")
    np.testing.assert_array_equal(whole_ids(scores, n_dev, k), want)


@pytest.mark.parametrize("path", [qsa.PATH_WARP, qsa.PATH_RADIX, qsa.PATH_SPLIT, qsa.PATH_SAMPLE])
def test_sharded_with_each_top_k_path(path):
    """Stage A may run any top-k path; the merged ids do not depend on it."""
    nq, C, k = 16, 6000, 32
    sc = inputs.normal_scores(7900, nq, C)
    n = np.full(nq, C, dtype=np.int32)
    scores = torch.from_numpy(sc).cuda()
    got, _, _ = sharded_ids(scores, torch.from_numpy(n).cuda(), k, [0, 1500, 3100, 4700, C], path=path)
    np.testing.assert_array_equal(got, oracle.select_f32(sc, n, k))


def test_merge_of_hand_written_candidates():
    """The merge on its own: scores and ids written by hand, with a tie across shards
    and empty slots; the result is the k first in (score descending, id ascending)."""
    k = 4
    cs = torch.tensor([[[5.0, 3.0, 1.0, -np.inf]], [[3.0, 4.0, 9.0, 0.0]]], dtype=torch.float32, device="cuda")
    ci = torch.tensor([[[10, 12, 14, -1]], [[2, 20, 30, 31]]], dtype=torch.int32, device="cuda")
    ids = torch.full((1, k), -7, dtype=torch.int32, device="cuda")
    qsa.merge_candidates(cs, ci, ids)
    # order: 9.0 (30), 5.0 (10), 4.0 (20), 3.0 tie: id 2 before id 12
    np.testing.assert_array_equal(ids.cpu().numpy(), [[2, 10, 20, 30]])
    # fewer candidates than k: all of them, ascending, then -1
    ci2 = torch.tensor([[[7, -1, -1, -1]], [[3, -1, -1, -1]]], dtype=torch.int32, device="cuda")
    qsa.merge_candidates(cs, ci2, ids)
    np.testing.assert_array_equal(ids.cpu().numpy(), [[3, 7, -1, -1]])


@pytest.mark.parametrize("G,k", [(128, 32), (4096, 1), (64, 64), (8, 512)])
def test_merge_at_its_capacity(G, k):
    """G x k = 4,096 candidates per query (the merge's capacity), on random lists with
    empty slots: the ids are the oracle's selection over the union of the lists."""
    nq = 6
    rng = np.random.default_rng(9700 + G + k)
    # distinct global ids; scores on a coarse grid so that ties across shards occur
    ids_all = rng.permutation(G * k * 4)[: G * k].reshape(G, 1, k).repeat(nq, axis=1).astype(np.int32)
    sc = (rng.integers(0, 50, size=(G, nq, k)) / 8.0).astype(np.float32)
    empty = rng.random((G, nq, k)) < 0.2
    ids_all = np.where(empty, -1, ids_all).astype(np.int32)
    sc = np.where(empty, -np.inf, sc).astype(np.float32)
    cs = torch.from_numpy(sc).cuda()
    ci = torch.from_numpy(ids_all).cuda()
    ids = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
    qsa.merge_candidates(cs, ci, ids)
    # the oracle's selection over dense rows that hold each candidate's score at its id
    # and -inf elsewhere (every row has far more than k candidates)
    n = G * k * 4
    rows = np.full((nq, n), -np.inf, dtype=np.float32)
    for qi in range(nq):
        v = ids_all[:, qi, :] >= 0
        rows[qi, ids_all[:, qi, :][v]] = sc[:, qi, :][v]
    want = oracle.select_f32(rows, np.full(nq, n, dtype=np.int32), k)
    np.testing.assert_array_equal(ids.cpu().numpy(), want)
