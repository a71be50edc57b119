"""GPU parity of the block top-k (qsa_block_topk) against the oracle, every path.

Scores are fed directly (continuous, 64-level, all-equal, negative, +-0), so
rule (a) is checked bit for bit on each forced path and on AUTO.
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

PATHS = [qsa.PATH_AUTO, qsa.PATH_RADIX, qsa.PATH_REGISTER, qsa.PATH_SAMPLE, qsa.PATH_SPLIT, qsa.PATH_WARP]


def run_topk(scores_np, n_blocks_np, k, path, active=-1, max_blocks=None, stride=None):
    nq, C = scores_np.shape
    stride = stride or C
    buf = torch.full((nq, stride), float("nan"), dtype=torch.float32, device="cuda")
    buf[:, :C] = torch.from_numpy(scores_np).cuda()
    mb = C if max_blocks is None else max_blocks
    n_dev = torch.from_numpy(np.ascontiguousarray(n_blocks_np, dtype=np.int32)).cuda()
    ids = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
    ws = qsa.alloc_workspace(nq, mb, k)
    qsa.block_topk(buf, n_dev, k, ids, ws, max_blocks=mb, active_blocks=active, path=path)
    flags = qsa.read_flags(ws)
    return ids.cpu().numpy(), flags, ws


def _supported(path, C, nq, k, active):
    bound = C if active < 0 else min(active, C)
    if path in (qsa.PATH_REGISTER, qsa.PATH_SAMPLE, qsa.PATH_WARP) and bound > 8192:
        return False
    if path == qsa.PATH_WARP and k > 32:
        return False
    return True


@pytest.mark.parametrize("path", PATHS, ids=[qsa.PATH_NAMES[p] for p in PATHS])
@pytest.mark.parametrize("kind", ["normal", "levels", "equal", "negative_zero"])
@pytest.mark.parametrize("shape", [(3, 4096, 4032, 32, -1), (256, 2048, 2048, 32, 2048),
                                   (16, 8192, 8125, 32, 8125), (7, 1000, 999, 5, -1)])
def test_topk_paths_match_oracle(path, kind, shape):
    nq, C, n, k, active = shape
    if not _supported(path, C, nq, k, active):
        pytest.skip("path cannot hold this row")
    seed = 6000 + C + nq
    if kind == "normal":
        sc = inputs.normal_scores(seed, nq, C)
    elif kind == "levels":
        sc = inputs.level_scores(seed, nq, C)
    elif kind == "equal":
        sc = np.full((nq, C), 0.75, dtype=np.float32)
    else:
        rng = np.random.default_rng(seed)
        sc = rng.choice(np.array([0.0, -0.0, -1.0, 2.0, -0.5], dtype=np.float32), size=(nq, C))
    nb = np.full(nq, n, dtype=np.int32)
    try:
        ids, flags, _ = run_topk(sc, nb, k, path, active=active)
    except qsa.QSAError as e:
        if e.status == qsa.ERR_UNSUPPORTED and path != qsa.PATH_AUTO:
            pytest.skip(f"forced path unsupported here: {e.reason}")
        raise
    want = oracle.select_f32(sc, nb, k)
    np.testing.assert_array_equal(ids, want)
    assert flags & qsa.ERROR_FLAGS == 0


@pytest.mark.parametrize("path", PATHS, ids=[qsa.PATH_NAMES[p] for p in PATHS])
def test_topk_edge_lengths(path):
    """n = 0, 1, k-1, k, k+1, ragged, capacity, and clamped n per query."""
    C, k = 4096, 32
    lens = [0, 1, 31, 32, 33, 64, 65, 127, 128, 129, 1000, 4095, 4096, 2049, 3, 4096]
    nq = len(lens)
    sc = inputs.normal_scores(6100, nq, C)
    nb = np.array(lens, dtype=np.int32)
    try:
        ids, flags, _ = run_topk(sc, nb, k, path)
    except qsa.QSAError as e:
        if e.status == qsa.ERR_UNSUPPORTED and path != qsa.PATH_AUTO:
            pytest.skip(e.reason)
        raise
    np.testing.assert_array_equal(ids, oracle.select_f32(sc, nb, k))
    assert flags & qsa.ERROR_FLAGS == 0


@pytest.mark.parametrize("path", PATHS, ids=[qsa.PATH_NAMES[p] for p in PATHS])
def test_topk_clamps_out_of_range_n_blocks(path):
    C, k = 2048, 16
    sc = inputs.normal_scores(6200, 4, C)
    nb = np.array([5000, -3, 100, 2048], dtype=np.int32)
    try:
        ids, flags, _ = run_topk(sc, nb, k, path)
    except qsa.QSAError as e:
        if e.status == qsa.ERR_UNSUPPORTED and path != qsa.PATH_AUTO:
            pytest.skip(e.reason)
        raise
    np.testing.assert_array_equal(ids, oracle.select_f32(sc, np.clip(nb, 0, C), k))
    assert flags & qsa.FLAG_NBLOCKS_CLAMPED


@pytest.mark.parametrize("k", [1, 2, 17, 64, 255, 1024])
@pytest.mark.parametrize("path", PATHS, ids=[qsa.PATH_NAMES[p] for p in PATHS])
def test_topk_k_range(path, k):
    nq, C = 5, 4000
    sc = inputs.level_scores(6300 + k, nq, C, levels=512)
    nb = np.array([4000, 3999, 1500, k, k + 1], dtype=np.int32)
    try:
        ids, flags, _ = run_topk(sc, nb, k, path, active=4000 if path == qsa.PATH_SAMPLE else -1)
    except qsa.QSAError as e:
        if e.status == qsa.ERR_UNSUPPORTED and path != qsa.PATH_AUTO:
            pytest.skip(e.reason)
        raise
    np.testing.assert_array_equal(ids, oracle.select_f32(sc, nb, k))


@pytest.mark.parametrize("path", [qsa.PATH_AUTO, qsa.PATH_RADIX, qsa.PATH_REGISTER, qsa.PATH_SAMPLE, qsa.PATH_WARP])
def test_topk_unaligned_stride_uses_scalar_loads(path):
    nq, C, k = 6, 3001, 32
    sc = inputs.normal_scores(6400, nq, C)
    nb = np.array([3001, 3000, 2999, 2998, 100, 40], dtype=np.int32)
    ids, flags, _ = run_topk(sc, nb, k, path, active=3001, stride=3003)
    np.testing.assert_array_equal(ids, oracle.select_f32(sc, nb, k))


def test_topk_large_capacity_radix_auto():
    """Rows past the on-chip paths (> 8,192 blocks) go to the radix kernel."""
    nq, C, k = 4, 20000, 32
    sc = inputs.normal_scores(6500, nq, C)
    nb = np.array([20000, 19999, 12345, 8193], dtype=np.int32)
    ids, flags, _ = run_topk(sc, nb, k, qsa.PATH_AUTO, active=20000)
    np.testing.assert_array_equal(ids, oracle.select_f32(sc, nb, k))
    assert qsa.auto_path(nq, C, 20000, k) == qsa.PATH_RADIX


def test_split_leaves_workspace_reusable_and_is_deterministic():
    nq, C, k = 3, 4096, 32
    sc = inputs.normal_scores(6600, nq, C)
    nb = np.array([4032, 4032, 626], dtype=np.int32)
    ids1, _, ws = run_topk(sc, nb, k, qsa.PATH_SPLIT)
    buf = torch.from_numpy(sc).cuda()
    ids = torch.empty((nq, k), dtype=torch.int32, device="cuda")
    n_dev = torch.from_numpy(nb).cuda()
    for _ in range(5):
        qsa.block_topk(buf, n_dev, k, ids, ws, path=qsa.PATH_SPLIT)
        np.testing.assert_array_equal(ids.cpu().numpy(), ids1)
    np.testing.assert_array_equal(ids1, oracle.select_f32(sc, nb, k))


def test_sample_fallback_is_taken_and_correct():
    """All-equal scores defeat the sampled bound (> 4,096 candidates): radix fallback."""
    nq, C, k = 8, 8192, 32
    sc = np.full((nq, C), 1.5, dtype=np.float32)
    sc[1, 5000] = 9.0
    nb = np.full(nq, 8192, dtype=np.int32)
    ids, flags, ws = run_topk(sc, nb, k, qsa.PATH_SAMPLE, active=8192)
    np.testing.assert_array_equal(ids, oracle.select_f32(sc, nb, k))
    assert flags & qsa.FLAG_SAMPLE_FALLBACK


def test_sample_filter_is_used_on_continuous_scores():
    """Continuous scores: the sampled bound keeps between k and 4,096 candidates for every query."""
    nq, C, k = 64, 8192, 32
    sc = inputs.normal_scores(6700, nq, C)
    nb = np.full(nq, 8125, dtype=np.int32)
    ids, flags, ws = run_topk(sc, nb, k, qsa.PATH_SAMPLE, active=8125)
    np.testing.assert_array_equal(ids, oracle.select_f32(sc, nb, k))
    assert flags == 0


@pytest.mark.parametrize("k", [1, 32, 100, 1024])
def test_sample_few_candidates_falls_back(k):
    """A spike per row: with k above the candidate count the filter falls back and stays exact."""
    nq, C = 6, 8192
    rng = np.random.default_rng(6800 + k)
    sc = rng.integers(0, 3, size=(nq, C)).astype(np.float32)
    sc[:, ::97] = 5.0
    nb = np.array([8192, 8191, 5000, 4097, 4096, 2000], dtype=np.int32)
    ids, flags, ws = run_topk(sc, nb, k, qsa.PATH_SAMPLE, active=8192)
    np.testing.assert_array_equal(ids, oracle.select_f32(sc, nb, k))
    assert flags & qsa.ERROR_FLAGS == 0


@pytest.mark.parametrize("nq", [4, 160])
@pytest.mark.parametrize("n", [33, 64, 65, 511, 512, 513, 1023, 1024, 1025, 2047, 2048, 4097, 8191, 8192])
@pytest.mark.parametrize("kind", ["normal", "levels", "equal"])
def test_warp_path_chunk_boundaries(nq, n, kind):
    """Rows that end inside, at and just past a warp's 1,024-block chunk (and half of it),
    for a few and for many queries, with continuous, quantised and all-equal scores (the
    last two take the radix fallbacks)."""
    C, k = 8192, 32
    seed = 6900 + n
    sc = (inputs.normal_scores(seed, nq, C) if kind == "normal" else
          inputs.level_scores(seed, nq, C) if kind == "levels" else np.full((nq, C), 0.5, dtype=np.float32))
    nb = np.resize(np.array([n, max(n - 1, 0), min(n + 1, C), n], dtype=np.int32), nq)
    ids, flags, _ = run_topk(sc, nb, k, qsa.PATH_WARP, active=C)
    np.testing.assert_array_equal(ids, oracle.select_f32(sc, nb, k))
    assert flags & qsa.ERROR_FLAGS == 0


def test_warp_path_rejects_large_k_and_long_rows():
    sc = inputs.normal_scores(6950, 2, 9000)
    nb = np.array([9000, 100], dtype=np.int32)
    with pytest.raises(qsa.QSAError) as e:
        run_topk(sc, nb, 32, qsa.PATH_WARP, active=9000)
    assert e.value.status == qsa.ERR_UNSUPPORTED
    with pytest.raises(qsa.QSAError) as e:
        run_topk(sc[:, :4096], np.array([4096, 100], dtype=np.int32), 33, qsa.PATH_WARP, active=4096)
    assert e.value.status == qsa.ERR_UNSUPPORTED
