"""Selection attention on the GPU against the FP64 oracle (parity rule (d)).

Small cases (bf16 and fp16) span several pair tiles, odd block counts, pads, ragged contexts
with partial tail blocks, k = 1 .. 64 (the one-CTA-per-SM form above 32), one
unit per CTA and units split over clusters, grids of more CTAs than the GPU holds,
several GQA groups, unsorted and repeated ids, ids past the context, NaN in the
cache rows past the context, empty token sets, and the ids the select path
itself produces.  The bench's configuration (256 queries x 64 heads in 4 GQA
groups, 520,000 tokens, k = 32) is checked on sampled queries.
"""
import numpy as np
import pytest

from workloads import inputs

from .parity import attn_to_device, attention_reference, check_rule_d, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def qsa():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from sparse_attention_kv_gb300 import qsa as q
    q.load()
    return q


def _run(qsa, case, ws=None, lse=True, ids=None, n_tokens=None):
    qa, kc, vt, d_ids, d_nt = attn_to_device(case)
    if ids is not None:
        d_ids = ids
    if n_tokens is not None:
        d_nt = n_tokens
    out = torch.full((case.nq, case.n_heads, 128), float("nan"), device="cuda")
    lse_t = torch.full((case.nq, case.n_heads), float("nan"), device="cuda") if lse else None
    qsa.select_attention(qa, kc, vt, d_ids, d_nt, out, lse_t, scale=case.scale, ws=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (lse_t.cpu().numpy() if lse else None)


def _ws(qsa):
    return torch.zeros(256, dtype=torch.uint8, device="cuda")


CASES = [
    # (seed, nq, n_kv, capacity, tokens, k, n_valid)
    (101, 1, 1, 4096, 4096, 32, None),
    (102, 16, 2, 8192, "ragged", 32, None),
    (103, 8, 1, 4096, 4000, 1, None),
    (104, 8, 3, 4096, "ragged", 7, None),
    (105, 6, 1, 8192, 8192, 64, None),
    (106, 6, 2, 8192, "ragged", 33, None),
    (107, 12, 1, 4096, 4096, 32, "random"),
    (108, 5, 4, 2048, "ragged", 16, None),
]


def _case(seed, nq, n_kv, cap, tokens, k, n_valid, dtype=inputs.BF16):
    if tokens == "ragged":
        tokens = inputs.ragged_tokens(seed, nq, cap // 64)
    if n_valid == "random":
        n_valid = np.random.default_rng(seed).integers(0, k + 1, size=nq)
    return inputs.make_attention_case(seed, nq, n_kv, cap, tokens, k, n_valid=n_valid, dtype=dtype)


@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.F16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("params", CASES, ids=[f"nq{c[1]}-kv{c[2]}-C{c[3]}-{c[4]}-k{c[5]}" for c in CASES])
def test_matches_oracle(qsa, params, dtype):
    c = _case(*params, dtype=dtype)
    ws = _ws(qsa)
    out, lse = _run(qsa, c, ws)
    ref, ref_lse, bounds = attention_reference(c)
    check_rule_d(out, lse, ref, ref_lse, bounds)
    assert qsa.read_flags(ws) == 0


WAVE_CASES = [
    # 320 units: more CTAs than the GPU holds at once (two per SM), with random pads
    # and empty rows among them
    (131, 80, 4, 4096, "ragged", 32, "random"),
    (132, 40, 8, 2048, "ragged", 7, None),
    # 80 units at k = 64: unsplit, one CTA per SM, all 512 TMEM columns for the logits
    (133, 80, 1, 8192, "ragged", 64, None),
]


@pytest.mark.parametrize("params", WAVE_CASES, ids=[f"nq{c[1]}-kv{c[2]}-k{c[5]}" for c in WAVE_CASES])
def test_more_units_than_resident_ctas_match_oracle(qsa, params):
    c = _case(*params)
    ws = _ws(qsa)
    out, lse = _run(qsa, c, ws)
    ref, ref_lse, bounds = attention_reference(c)
    check_rule_d(out, lse, ref, ref_lse, bounds)
    assert qsa.read_flags(ws) == 0


def test_split_and_unsplit_forms_both_match(qsa):
    """80 queries x 2 KV heads fill the GPU (one CTA per unit); 4 of them alone are
    split over clusters of CTAs that combine their partials: both match the oracle."""
    c = _case(109, 80, 2, 4096, "ragged", 32, None)
    full, full_lse = _run(qsa, c)
    rows = np.arange(4)
    sub = inputs.AttnCase(qa=c.qa[rows], kc=c.kc, vc=c.vc, ids=c.ids[rows], n_tokens=c.n_tokens[rows],
                          scale=c.scale)
    part, part_lse = _run(qsa, sub)
    ref, ref_lse, bounds = attention_reference(c, rows)
    check_rule_d(full[rows], full_lse[rows], ref, ref_lse, bounds)
    check_rule_d(part, part_lse, ref, ref_lse, bounds)
    assert not np.array_equal(part, full[rows])   # two different reductions


def test_without_lse_or_workspace_the_output_is_the_same(qsa):
    c = _case(*CASES[1])
    a, _ = _run(qsa, c, _ws(qsa))
    b, _ = _run(qsa, c, None, lse=False)
    np.testing.assert_array_equal(a, b)


def test_unsorted_repeated_and_out_of_context_ids(qsa):
    c = _case(111, 8, 2, 4096, "ragged", 32, 24)
    rng = np.random.default_rng(5)
    ids = c.ids.copy()
    nb = inputs.blocks_for_tokens(c.n_tokens)
    for q in range(c.nq):
        row = ids[q]
        m = int((row >= 0).sum())
        row[m:m + 3] = [row[0], nb[q] + 5, -7]     # a repeat, one past the context, a negative
        ids[q] = rng.permutation(row)
    c.ids = ids
    ws = _ws(qsa)
    out, lse = _run(qsa, c, ws)
    ref, ref_lse, bounds = attention_reference(c)
    check_rule_d(out, lse, ref, ref_lse, bounds)
    assert qsa.read_flags(ws) == qsa.FLAG_BAD_ID


@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.F16], ids=["bf16", "fp16"])
def test_cache_rows_past_the_context_take_no_part(qsa, dtype):
    """NaN in every K and V row at or past each query's context: outputs unchanged, bit for bit."""
    n = 64 * 37 + 23                                   # a partial tail block
    c = inputs.make_attention_case(112, 8, 1, 4096, n, 32, dtype=dtype)
    base = inputs.random_ids(113, np.full(8, 37), 31)
    for q in range(8):                                 # 31 blocks below the tail, then the tail block
        v = base[q][base[q] >= 0]
        c.ids[q] = np.r_[v, 37, np.full(31 - len(v), -1)]
    clean, clean_lse = _run(qsa, c)
    nan = np.uint16(0x7E00 if dtype == inputs.F16 else 0x7FC0)
    c.kc = c.kc.copy()
    c.vc = c.vc.copy()
    c.kc[:, n:] = nan
    c.vc[:, n:] = nan
    dirty, dirty_lse = _run(qsa, c)
    np.testing.assert_array_equal(dirty, clean)
    np.testing.assert_array_equal(dirty_lse, clean_lse)
    ref, ref_lse, bounds = attention_reference(c)
    check_rule_d(dirty, dirty_lse, ref, ref_lse, bounds)


def test_empty_token_sets(qsa):
    c = _case(114, 4, 2, 2048, 2048, 8, None)
    c.ids[0] = -1                     # pads only
    c.n_tokens[1] = 0                 # no context (its ids are then out of context)
    c.ids[2] = -1
    c.ids[2, 0] = 31                  # in context
    ws = _ws(qsa)
    out, lse = _run(qsa, c, ws)
    ref, ref_lse, bounds = attention_reference(c)
    assert np.isneginf(ref_lse[:2]).all()
    check_rule_d(out, lse, ref, ref_lse, bounds)
    assert qsa.read_flags(ws) == qsa.FLAG_BAD_ID


def test_context_past_capacity_is_clamped(qsa):
    c = _case(115, 4, 1, 2048, 2048, 8, None)
    c.n_tokens[2] = 10 ** 6
    ws = _ws(qsa)
    out, lse = _run(qsa, c, ws)
    c.n_tokens[2] = 2048
    ref, ref_lse, bounds = attention_reference(c)
    check_rule_d(out, lse, ref, ref_lse, bounds)
    assert qsa.read_flags(ws) == qsa.FLAG_NBLOCKS_CLAMPED


def test_on_the_ids_of_the_select_path(qsa):
    """Select (chained and fused) on a 131,072-token prompt, then attend over those ids."""
    sc = inputs.make_case(116, 64, 16, 2048, inputs.BF16, 131_072, 32, active_blocks=2048)
    q, w, kb, nb = to_device(sc)
    ws = qsa.alloc_workspace(64, 2048, 32, fused=True)
    ids_c = torch.empty((64, 32), dtype=torch.int32, device="cuda")
    ids_f = torch.empty_like(ids_c)
    scores = torch.empty((64, 2048), dtype=torch.float32, device="cuda")
    qsa.select(q, w, kb, nb, 32, ids_c, ws, scores=scores, active_blocks=2048)
    qsa.select(q, w, kb, nb, 32, ids_f, ws, fused=True, active_blocks=2048)
    assert torch.equal(ids_c, ids_f)
    ids = ids_c.cpu().numpy()
    c = inputs.make_attention_case(117, 64, 4, 131_072, sc.tokens, 32, ids=ids)
    out, lse = _run(qsa, c, ids=ids_c)
    rows = np.arange(0, 64, 4)
    ref, ref_lse, bounds = attention_reference(c, rows)
    check_rule_d(out[rows], lse[rows], ref, ref_lse, bounds)


PATHS_B2B = ["auto", "split", "sample", "register", "radix", "warp"]


@pytest.mark.parametrize("path", PATHS_B2B)
@pytest.mark.parametrize("nq,fused", [(3, False), (3, True), (64, False), (64, True)])
def test_select_then_attention_back_to_back(qsa, nq, fused, path):
    """The attention enqueued right behind the select that writes its ids (no host step
    between, so it launches as the programmatic dependent of whichever top-k kernel
    wrote them)."""
    if fused and path != "auto":
        pytest.skip("the fused form takes the auto path only")
    path_code = {"auto": qsa.PATH_AUTO, "split": qsa.PATH_SPLIT, "sample": qsa.PATH_SAMPLE,
                 "register": qsa.PATH_REGISTER, "radix": qsa.PATH_RADIX, "warp": qsa.PATH_WARP}[path]
    sc = inputs.make_case(118 + nq, nq, 16, 2048, inputs.BF16, 131_072, 32, active_blocks=-1 if nq == 3 else 2048)
    q, w, kb, nb = to_device(sc)
    c = inputs.make_attention_case(119 + nq, nq, 4, 131_072, sc.tokens, 32)
    qa, kc, vt, _, nt = attn_to_device(c)
    ws = qsa.alloc_workspace(nq, 2048, 32, fused=True)
    ids = torch.full((nq, 32), -9, dtype=torch.int32, device="cuda")
    scores = None if fused else torch.empty((nq, 2048), dtype=torch.float32, device="cuda")
    out = torch.full((nq, c.n_heads, 128), float("nan"), device="cuda")
    lse = torch.full((nq, c.n_heads), float("nan"), device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):   # repeated: every call's attention follows its own select
        ids.fill_(-9)
        try:
            qsa.select(q, w, kb, nb, 32, ids, ws, scores=scores, fused=fused, active_blocks=sc.active_blocks,
                       path=path_code)
        except qsa.QSAError as e:
            if e.status == qsa.ERR_UNSUPPORTED:
                pytest.skip(f"{path} does not take this shape")
            raise
        qsa.select_attention(qa, kc, vt, ids, nt, out, lse, scale=c.scale, ws=ws)
    torch.cuda.synchronize()
    assert qsa.read_flags(ws) & qsa.ERROR_FLAGS == 0
    c.ids = ids.cpu().numpy()
    rows = np.arange(nq) if nq <= 8 else np.arange(0, nq, 8)
    ref, ref_lse, bounds = attention_reference(c, rows)
    check_rule_d(out.cpu().numpy()[rows], lse.cpu().numpy()[rows], ref, ref_lse, bounds)


@pytest.mark.parametrize("dtype", [inputs.BF16, inputs.F16], ids=["bf16", "fp16"])
def test_vcache_transpose_is_the_block_transpose(qsa, dtype):
    """The library's layout conversion, bit for bit, in full and over a block range."""
    c = inputs.make_attention_case(140, 1, 3, 4096, 4096, 1, dtype=dtype)
    tdt = torch.float16 if dtype == inputs.F16 else torch.bfloat16
    v = torch.from_numpy(c.vc.view(np.int16)).view(tdt).cuda()
    want = inputs.vcache_blocks_transposed(c.vc)
    vt = torch.zeros((3, 64, 128, 64), dtype=tdt, device="cuda")
    qsa.vcache_transpose(v, vt)
    np.testing.assert_array_equal(vt.cpu().view(torch.int16).numpy().view(np.uint16), want)
    vt.zero_()
    qsa.vcache_transpose(v, vt, first_block=10, n_blocks=7)
    got = vt.cpu().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got[:, 10:17], want[:, 10:17])
    assert (got[:, :10] == 0).all() and (got[:, 17:] == 0).all()


@pytest.fixture(scope="module")
def deep_attention():
    """The bench's configuration: 256 queries x 64 heads (4 GQA groups of 16),
    capacity 524,288 tokens, contexts of 520,000 tokens, k = 32 random blocks."""
    return inputs.deep_attention_case()


def test_deep_prompt_sampled_queries(qsa, deep_attention):
    c = deep_attention
    ws = _ws(qsa)
    out, lse = _run(qsa, c, ws)
    rows = np.array([0, 1, 77, 128, 200, 255])
    ref, ref_lse, bounds = attention_reference(c, rows)
    check_rule_d(out[rows], lse[rows], ref, ref_lse, bounds)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert qsa.read_flags(ws) == 0
