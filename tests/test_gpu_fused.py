"""GPU parity of the fused score-then-select (qsa_select with fused = 1).

The fused kernel computes the same scores as the chained scorer and selects on
chip, so its ids must equal the chained path's ids bit for bit, and its
optional debug copy of the scores must equal the chained scores bit for bit;
both are also checked against the oracle (rules (a) and (c)).
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


def run(case, fused, with_scores=True, ws=None, active=None):
    q, w, kb, nb = parity.to_device(case)
    act = case.active_blocks if active is None else active
    sc = None
    if with_scores or not fused:
        sc = torch.full((case.nq, case.max_blocks), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((case.nq, case.k), -7, dtype=torch.int32, device="cuda")
    if ws is None:
        ws = qsa.alloc_workspace(case.nq, case.max_blocks, case.k, fused=fused)
    qsa.select(q, w, kb, nb, case.k, ids, ws, scores=sc, fused=fused, active_blocks=act)
    flags = qsa.read_flags(ws)
    assert flags & qsa.ERROR_FLAGS == 0, f"device flags {flags:#x}"
    return ids.cpu().numpy(), (sc.cpu().numpy() if sc is not None else None), ws


def check_fused_equals_chained(case, active=None):
    ids_c, sc_c, _ = run(case, fused=False, active=active)
    ids_f, sc_f, _ = run(case, fused=True, active=active)
    np.testing.assert_array_equal(ids_f, ids_c)
    for qi, n in enumerate(case.n_blocks):
        np.testing.assert_array_equal(sc_f[qi, :n], sc_c[qi, :n])
    parity.check_rule_a(ids_f, oracle.select_f32(sc_f, case.n_blocks, case.k))
    return ids_f, sc_f


def test_fused_tiny_fp32():
    check_fused_equals_chained(inputs.tiny_case())


@pytest.mark.parametrize("i", range(len(inputs.DECODE_TOKENS)))
def test_fused_decode(i):
    case = inputs.decode_case(i)
    ids, sc = check_fused_equals_chained(case)
    ref = oracle.block_scores(case.q, case.w, case.kblk, case.n_blocks, case.dtype)
    parity.check_rule_c(ids, ref, oracle.select(ref, case.n_blocks, case.k), case.n_blocks, case.k, case.dtype)


def test_fused_prompt():
    check_fused_equals_chained(inputs.prompt_case())


@pytest.mark.parametrize("i", range(len(inputs.DEEP_TOKENS)))
def test_fused_deep(i):
    case = inputs.deep_case(i)
    ids, sc = check_fused_equals_chained(case)
    ref = oracle.block_scores(case.q, case.w, case.kblk, case.n_blocks, case.dtype)
    parity.check_rule_c(ids, ref, oracle.select(ref, case.n_blocks, case.k), case.n_blocks, case.k, case.dtype)


@pytest.mark.parametrize("kind", ["equal_kblk", "w_zero", "ragged"])
def test_fused_stress(kind):
    case = inputs.stress_case(kind)
    ids, _ = check_fused_equals_chained(case)
    if kind in ("equal_kblk", "w_zero"):
        np.testing.assert_array_equal(ids, np.tile(np.arange(case.k, dtype=np.int32), (case.nq, 1)))


@pytest.mark.parametrize("H", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("dtype", [inputs.F32, inputs.BF16, inputs.E4M3])
def test_fused_heads_dtypes_and_short_rows(H, dtype):
    """Every head count and input type; ragged rows including n = 0, 1, k-1, k, k+1."""
    nq, C, k = 37, 700, 24
    toks = inputs.ragged_tokens(8000 + H, nq, C)
    toks[:6] = [0, 1, 64 * (k - 1), 64 * k, 64 * k + 1, 64 * C]
    case = inputs.make_case(8000 + H + 10 * dtype, nq, H, C, dtype, toks, k, active_blocks=C)
    check_fused_equals_chained(case)


@pytest.mark.parametrize("k", [1, 7, 64, 200])
def test_fused_k_range(k):
    case = inputs.make_case(8100 + k, 40, 16, 3000, inputs.BF16, inputs.ragged_tokens(8100 + k, 40, 3000), k,
                            active_blocks=3000)
    check_fused_equals_chained(case)


def test_fused_many_queries_several_waves_and_no_active_count():
    case = inputs.make_case(8200, 700, 16, 1500, inputs.BF16, inputs.ragged_tokens(8200, 700, 1500), 32)
    check_fused_equals_chained(case, active=-1)


def test_fused_without_scores_and_workspace_reuse():
    case = inputs.deep_case(2)
    ids_c, _, _ = run(case, fused=False)
    ids1, none, ws = run(case, fused=True, with_scores=False)
    assert none is None
    np.testing.assert_array_equal(ids1, ids_c)
    for _ in range(3):   # the same workspace serves the next calls (no state carries over)
        ids2, _, _ = run(case, fused=True, with_scores=False, ws=ws)
        np.testing.assert_array_equal(ids2, ids_c)


def test_fused_large_k_long_rows_takes_more_tiles_per_cta():
    """k = 1,024 over 60,000 blocks: the merge holds at most 4,096 candidates per query,
    so the fused form gives each CTA more tiles (and fewer CTAs per query)."""
    case = inputs.make_case(8300, 4, 16, 60000, inputs.BF16, 64 * 60000, 1024, active_blocks=60000)
    ids_c, _, _ = run(case, fused=False)
    ids_f, _, _ = run(case, fused=True, with_scores=False)
    np.testing.assert_array_equal(ids_f, ids_c)


def test_fused_rejects_shapes_that_do_not_fit_and_forced_paths():
    # 100,000 blocks at k = 1,024: four CTAs per query at most, each would hold more
    # scores than its shared memory
    case = inputs.make_case(8301, 4, 16, 100000, inputs.BF16, 64 * 100000, 1024, active_blocks=100000)
    with pytest.raises(qsa.QSAError) as e:
        run(case, fused=True, with_scores=False)
    assert e.value.status == qsa.ERR_UNSUPPORTED
    small = inputs.decode_case(0)
    q, w, kb, nb = parity.to_device(small)
    ids = torch.empty((small.nq, small.k), dtype=torch.int32, device="cuda")
    ws = qsa.alloc_workspace(small.nq, small.max_blocks, small.k, fused=True)
    with pytest.raises(qsa.QSAError) as e:
        qsa.select(q, w, kb, nb, small.k, ids, ws, fused=True, path=qsa.PATH_SAMPLE)
    assert e.value.status == qsa.ERR_UNSUPPORTED
    # the fused form's candidate lists need the fused workspace size
    small_ws = qsa.alloc_workspace(small.nq, small.max_blocks, small.k)
    with pytest.raises(qsa.QSAError) as e:
        qsa.select(q, w, kb, nb, small.k, ids, small_ws, fused=True)
    assert e.value.status == qsa.ERR_WORKSPACE
