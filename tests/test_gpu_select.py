"""GPU parity of the scorer and of the whole select path on the five workloads.

Rule (b) on the scores, rule (a) on the top-k of the GPU's own scores, rule (c)
end to end against the FP64 oracle (see tests/parity.py).
"""
import numpy as np
import pytest

import oracle
from workloads import inputs
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from sparse_attention_kv_gb300 import qsa  # noqa: E402


def gpu_scores(case, active=None):
    q, w, kb, nb = parity.to_device(case)
    act = case.active_blocks if active is None else active
    sc = torch.full((case.nq, case.max_blocks), float("nan"), dtype=torch.float32, device="cuda")
    ws = qsa.alloc_workspace(case.nq, case.max_blocks, case.k)
    qsa.block_scores(q, w, kb, nb, sc, active_blocks=act, ws=ws)
    flags = qsa.read_flags(ws)
    return sc.cpu().numpy(), flags


def run_select(case, path=qsa.PATH_AUTO, fused=False):
    q, w, kb, nb = parity.to_device(case)
    sc = torch.full((case.nq, case.max_blocks), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((case.nq, case.k), -7, dtype=torch.int32, device="cuda")
    ws = qsa.alloc_workspace(case.nq, case.max_blocks, case.k, fused=fused)
    qsa.select(q, w, kb, nb, case.k, ids, ws, scores=sc, fused=fused,
               active_blocks=case.active_blocks, path=path)
    flags = qsa.read_flags(ws)
    return ids.cpu().numpy(), sc.cpu().numpy(), flags


def full_check(case, path=qsa.PATH_AUTO):
    ref = oracle.block_scores(case.q, case.w, case.kblk, case.n_blocks, case.dtype)
    ref_ids = oracle.select(ref, case.n_blocks, case.k)
    ids, sc, flags = run_select(case, path)
    assert flags & qsa.ERROR_FLAGS == 0, f"device flags {flags:#x}"
    # scores are written exactly for b < n and left alone past it
    for qi, n in enumerate(case.n_blocks):
        assert np.isfinite(sc[qi, :n]).all()
        assert np.isnan(sc[qi, n:]).all()
    err = parity.check_rule_b(sc, ref, case.n_blocks, case.dtype)
    parity.check_rule_a(ids, oracle.select_f32(sc, case.n_blocks, case.k))
    r = parity.check_rule_c(ids, ref, ref_ids, case.n_blocks, case.k, case.dtype, tight_tol=4 * max(err, 1e-9))
    print(f"{case.name}: max score err {err:.2e}; rule (c) {r['exact']}/{r['queries']} exact, "
          f"{r['excused']} excused, near-ties {r['near_tie']} (tight {r['near_tie_tight']})")
    return ids, sc, r


def test_tiny_fp32():
    full_check(inputs.tiny_case())


@pytest.mark.parametrize("i", range(len(inputs.DECODE_TOKENS)))
def test_decode_window(i):
    full_check(inputs.decode_case(i))


def test_prompt():
    full_check(inputs.prompt_case())


@pytest.mark.parametrize("i", range(len(inputs.DEEP_TOKENS)))
def test_deep_prompt(i):
    full_check(inputs.deep_case(i))


@pytest.mark.parametrize("kind", ["equal_kblk", "w_zero", "ragged"])
def test_stress_end_to_end(kind):
    case = inputs.stress_case(kind)
    ids, sc, r = full_check(case)
    if kind in ("equal_kblk", "w_zero"):
        # every score ties: the lowest block ids, exactly, no excusal
        assert r["exact"] == r["queries"]
        want = np.minimum(case.n_blocks[:, None], case.k)
        np.testing.assert_array_equal(ids, np.tile(np.arange(case.k, dtype=np.int32), (case.nq, 1)))


@pytest.mark.parametrize("path", [qsa.PATH_RADIX, qsa.PATH_REGISTER, qsa.PATH_SAMPLE, qsa.PATH_SPLIT, qsa.PATH_WARP])
def test_every_path_end_to_end_on_decode_and_prompt(path):
    for case in (inputs.decode_case(1), inputs.prompt_case()):
        try:
            full_check(case, path)
        except qsa.QSAError as e:
            if e.status != qsa.ERR_UNSUPPORTED:
                raise


@pytest.mark.parametrize("fused", [False, True])
def test_e4m3_decode_window_chained_and_fused(fused):
    case = inputs.decode_e4m3_case()
    ref = oracle.block_scores(case.q, case.w, case.kblk, case.n_blocks, case.dtype)
    ids, sc, flags = run_select(case, fused=fused)
    assert flags & qsa.ERROR_FLAGS == 0
    err = parity.check_rule_b(sc, ref, case.n_blocks, case.dtype)
    assert err <= 1e-5, f"e4m3 products are exact in fp32: error {err:.2e} is above fp32 rounding"
    parity.check_rule_a(ids, oracle.select_f32(sc, case.n_blocks, case.k))
    r = parity.check_rule_c(ids, ref, oracle.select(ref, case.n_blocks, case.k), case.n_blocks, case.k, case.dtype)
    assert r["excused"] == 0 and r["exact"] == case.nq


def test_e4m3_deep_prompt_sampled():
    """fp8 q and kblk at 520,000 tokens: scores and ids of 32 sampled queries against
    the oracle, both select forms, and the fused ids equal to the chained ones."""
    case = inputs.deep_e4m3_case()
    ids, sc, flags = run_select(case)
    assert flags & qsa.ERROR_FLAGS == 0
    fids, fsc, fflags = run_select(case, fused=True)
    assert fflags & qsa.ERROR_FLAGS == 0
    np.testing.assert_array_equal(fids, ids)
    rows = np.arange(0, 256, 8)
    sub = inputs.Case(q=case.q[rows], w=case.w[rows], kblk=case.kblk, n_blocks=case.n_blocks[rows],
                      tokens=case.tokens[rows], dtype=case.dtype, k=case.k, active_blocks=case.active_blocks)
    ref = oracle.block_scores(sub.q, sub.w, sub.kblk, sub.n_blocks, sub.dtype)
    err = parity.check_rule_b(sc[rows], ref, sub.n_blocks, sub.dtype)
    assert err <= 1e-5, f"e4m3 products are exact in fp32: error {err:.2e} is above fp32 rounding"
    parity.check_rule_a(ids[rows], oracle.select_f32(sc[rows], sub.n_blocks, sub.k))
    r = parity.check_rule_c(ids[rows], ref, oracle.select(ref, sub.n_blocks, sub.k), sub.n_blocks, sub.k,
                            sub.dtype)
    assert r["excused"] == 0 and r["exact"] == len(rows)


@pytest.mark.parametrize("H", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("dtype", [inputs.F32, inputs.BF16, inputs.E4M3])
def test_scorer_heads_and_dtypes(H, dtype):
    """Every head count, every input type, a group split across CTAs and a ragged tail."""
    nq = 37
    toks = inputs.ragged_tokens(7000 + H, nq, 300)
    case = inputs.make_case(7000 + H + 10 * dtype, nq, H, 300, dtype, toks, 8, active_blocks=300)
    sc, flags = gpu_scores(case)
    assert flags & qsa.ERROR_FLAGS == 0
    ref = oracle.block_scores(case.q, case.w, case.kblk, case.n_blocks, case.dtype)
    parity.check_rule_b(sc, ref, case.n_blocks, case.dtype)
    for qi, n in enumerate(case.n_blocks):
        assert np.isnan(sc[qi, n:]).all()


def test_scorer_active_count_never_changes_scores():
    case = inputs.decode_case(5)
    a, _ = gpu_scores(case, active=-1)
    b, _ = gpu_scores(case, active=4032)
    np.testing.assert_array_equal(a[:, :4032], b[:, :4032])


def test_scorer_clamps_n_blocks_to_active_bound():
    case = inputs.make_case(7100, 4, 16, 1024, inputs.BF16, [64 * 500, 64 * 1024, 64 * 10, 64], 32)
    sc, flags = gpu_scores(case, active=600)
    assert flags & qsa.FLAG_NBLOCKS_CLAMPED
    assert np.isfinite(sc[1, :600]).all() and np.isnan(sc[1, 600:]).all()


def test_select_is_deterministic():
    case = inputs.deep_case(0)
    a = run_select(case)
    b = run_select(case)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("nq,H", [(100, 16), (200, 8)])
def test_scorer_many_groups_partial_group_ragged_and_clamped(nq, H):
    """Many query groups with a partial last one, contexts from 0 to the full 8,192 blocks
    and two out of range: scores against FP64 (rule b), untouched past n, the clamp
    flag raised."""
    C = 8192
    toks = inputs.ragged_tokens(7300 + nq, nq, C)
    toks[:6] = [0, 64, 64 * 128, 64 * 128 + 1, 64 * C, 64 * C - 63]
    case = inputs.make_case(7300 + nq + H, nq, H, C, inputs.BF16, toks, 32, active_blocks=C)
    q, w, kb, nb = parity.to_device(case)
    nb[7] = C + 500      # past the bound: clamped to it
    nb[8] = -4           # negative: clamped to 0
    sc = torch.full((nq, C), float("nan"), dtype=torch.float32, device="cuda")
    ws = qsa.alloc_workspace(nq, C, 32)
    qsa.block_scores(q, w, kb, nb, sc, active_blocks=C, ws=ws)
    flags = qsa.read_flags(ws)
    assert flags & qsa.FLAG_NBLOCKS_CLAMPED
    assert flags & qsa.FLAG_WAIT_TIMEOUT == 0
    n_eff = np.clip(nb.cpu().numpy(), 0, C)
    got = sc.cpu().numpy()
    ref = oracle.block_scores(case.q, case.w, case.kblk, n_eff, case.dtype)
    parity.check_rule_b(got, ref, n_eff, case.dtype)
    for qi, n in enumerate(n_eff):
        assert np.isnan(got[qi, n:]).all()


def test_fp32_inputs_at_scale_chained_and_fused():
    """fp32 q and kblk (the three-term TF32 split) at 64 queries x 2,048 blocks with ragged
    contexts: scores within 1e-4 of FP64 (rule b), ids by rules (a) and (c), and the fused
    form's ids equal to the chained form's."""
    nq, C, k = 64, 2048, 32
    toks = inputs.ragged_tokens(7400, nq, C)
    case = inputs.make_case(7400, nq, 16, C, inputs.F32, toks, k, active_blocks=C)
    ids, sc, r = full_check(case)
    ids_f, _, flags = run_select(case, fused=True)
    assert flags & qsa.ERROR_FLAGS == 0
    np.testing.assert_array_equal(ids_f, ids)


@pytest.mark.parametrize("path", [qsa.PATH_WARP, qsa.PATH_SAMPLE, qsa.PATH_REGISTER, qsa.PATH_RADIX])
def test_every_path_end_to_end_on_the_deep_prompt(path):
    """The 256-query, 520,000-token prompt through each top-k path that holds its rows."""
    full_check(inputs.deep_case(2), path)


@pytest.mark.parametrize("fused", [False, True])
def test_back_to_back_selects_share_the_scores_buffer(fused):
    """Two chained selects enqueued back to back with no host step between them, on one
    scores buffer and one workspace: the second call's scorer is a programmatic
    dependent of the first call's top-k (which lets dependents launch at its entry), so
    it must not read its inputs or overwrite the scores before that top-k has read them
    (fused: the next scorer's candidate lists wait for the merge before them).  Each
    call's ids must be the oracle's selection over its own scores."""
    a, b = inputs.deep_case(0), inputs.deep_case(2)
    qa, wa, kba, nba = parity.to_device(a)
    qb, wb, kbb, nbb = parity.to_device(b)
    C = a.max_blocks
    ws = qsa.alloc_workspace(a.nq, C, a.k, fused=fused)
    ref = []
    for q, w, kb, nb, case in ((qa, wa, kba, nba, a), (qb, wb, kbb, nbb, b)):
        sc = torch.empty((case.nq, C), device="cuda")
        qsa.block_scores(q, w, kb, nb, sc, active_blocks=case.active_blocks, ws=ws)
        torch.cuda.synchronize()
        ref.append(oracle.select_f32(sc.cpu().numpy(), nb.cpu().numpy(), case.k))
    shared = torch.full((a.nq, C), float("nan"), device="cuda")
    outs = [torch.full((a.nq, a.k), -7, dtype=torch.int32, device="cuda") for _ in range(10)]
    for i, ids in enumerate(outs):
        q, w, kb, nb, case = (qa, wa, kba, nba, a) if i % 2 == 0 else (qb, wb, kbb, nbb, b)
        qsa.select(q, w, kb, nb, case.k, ids, ws, scores=shared, fused=fused, active_blocks=case.active_blocks)
    torch.cuda.synchronize()
    assert qsa.read_flags(ws) & qsa.ERROR_FLAGS == 0
    for i, ids in enumerate(outs):
        np.testing.assert_array_equal(ids.cpu().numpy(), ref[i % 2], err_msg=f"call {i}")
