"""Pins of the CPU oracle against facts fixed outside it.

Each test checks the oracle against something other than itself: hand-worked
fixtures (tests/golden), identities of the ReLU/weighted-sum structure that a
library matmul can check, an exactly rounded sum, brute force over all
k-subsets, and closed forms of the tie rule.  A mutation test at the end
plants plausible mistakes in a copy of the oracle and checks that the pins
catch every one.
"""
import itertools
import json
import math
import os
import shutil
import subprocess
import ctypes

import numpy as np
import pytest

import oracle
from workloads import inputs


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- scores

def test_scores_hand_fixture(golden_dir):
    g = _load(golden_dir, "scores_hand.json")
    q = np.array(g["q"], dtype=np.float32)
    w = np.array(g["w"], dtype=np.float32)
    kb = np.array(g["kblk"], dtype=np.float32)
    n = np.array(g["n_blocks"], dtype=np.int32)
    s = oracle.block_scores(q, w, kb, n)
    np.testing.assert_array_equal(s, np.array(g["scores"], dtype=np.float64))
    for k, want in g["select"].items():
        np.testing.assert_array_equal(oracle.select(s, n, int(k)), np.array(want))


def test_bf16_widening_fixture(golden_dir):
    g = _load(golden_dir, "bf16_hand.json")
    D = g["head_dim"]
    q = np.zeros((1, 1, D), dtype=np.uint16)
    q[0, 0, 0] = int(g["q_bits_d0"], 16)
    kb = np.zeros((len(g["kblk_bits_d0"]), D), dtype=np.uint16)
    for b, hx in enumerate(g["kblk_bits_d0"]):
        kb[b, 0] = int(hx, 16)
    w = np.array([[g["w"]]], dtype=np.float32)
    n = np.array([kb.shape[0]], dtype=np.int32)
    s = oracle.block_scores(q, w, kb, n, oracle.BF16)
    np.testing.assert_array_equal(s[0], np.array(g["scores"]))


def _rand_case(seed, nq=3, H=4, D=128, C=37, dtype=inputs.F32):
    c = inputs.make_case(seed, nq, H, C, dtype, C * 64, 8)
    if D != 128:
        rng = np.random.default_rng(seed + 1)
        c.q = rng.standard_normal((nq, H, D)).astype(np.float32)
        c.kblk = rng.standard_normal((C, D)).astype(np.float32)
    return c


def test_relu_per_head_identities():
    """s(q) + s(-q) = sum_h w|q_h.k| and s(q) - s(-q) = (sum_h w_h q_h).k (matmul)."""
    c = _rand_case(11, nq=4, H=5, C=50)
    n = np.full(c.nq, c.max_blocks, dtype=np.int32)
    sp = oracle.block_scores(c.q, c.w, c.kblk, n)
    sm = oracle.block_scores(-c.q, c.w, c.kblk, n)
    dots = np.einsum("qhd,bd->qhb", c.q.astype(np.float64), c.kblk.astype(np.float64))
    abs_sum = np.einsum("qh,qhb->qb", c.w.astype(np.float64), np.abs(dots))
    lin = (c.w.astype(np.float64)[:, :, None] * c.q.astype(np.float64)).sum(1) @ \
        c.kblk.astype(np.float64).T
    scale = np.abs(abs_sum).max()
    assert np.abs((sp + sm) - abs_sum).max() <= 1e-12 * scale
    assert np.abs((sp - sm) - lin).max() <= 1e-12 * scale


def test_linear_in_w_and_homogeneous_in_q():
    c = _rand_case(12, nq=2, H=3, C=20)
    n = np.full(c.nq, c.max_blocks, dtype=np.int32)
    rng = np.random.default_rng(5)
    w2 = rng.random(c.w.shape).astype(np.float32)
    s1 = oracle.block_scores(c.q, c.w, c.kblk, n)
    s2 = oracle.block_scores(c.q, w2, c.kblk, n)
    s12 = oracle.block_scores(c.q, (c.w + w2).astype(np.float32), c.kblk, n)
    # w + w2 in fp32 is exact only up to rounding of the sum; compare in that light
    assert np.abs(s12 - (s1 + s2)).max() <= 1e-6 * np.abs(s12).max()
    s_half = oracle.block_scores((c.q * np.float32(0.5)), c.w, c.kblk, n)   # exact scaling
    np.testing.assert_allclose(s_half, 0.5 * s1, rtol=0, atol=1e-12 * np.abs(s1).max())


def test_exactly_rounded_sum_crosscheck():
    """Products of fp32 inputs are exact in double; compare with math.fsum of them."""
    c = inputs.tiny_case()
    s = oracle.block_scores(c.q, c.w, c.kblk, c.n_blocks)
    q64 = c.q.astype(np.float64)
    k64 = c.kblk.astype(np.float64)
    w64 = c.w.astype(np.float64)
    worst = 0.0
    for b in range(c.max_blocks):
        terms = []
        for h in range(c.n_heads):
            dot = math.fsum((q64[0, h] * k64[b]).tolist())
            terms.append(w64[0, h] * max(dot, 0.0))
        ref = math.fsum(terms)
        worst = max(worst, abs(ref - s[0, b]))
    assert worst <= 1e-13 * np.abs(s).max()


def _e4m3_values(codes):
    """Values of e4m3 codes read through the scorer: one head, w = 1, q = +-1 on d0,
    the codes in kblk[:, 0]; relu(q.k) for q = +1 and q = -1 give the value's two sides."""
    kb = np.zeros((len(codes), 128), dtype=np.uint8)
    kb[:, 0] = codes
    n = np.array([len(codes)], np.int32)
    w = np.ones((1, 1), np.float32)
    pos, neg = np.zeros((1, 1, 128), np.uint8), np.zeros((1, 1, 128), np.uint8)
    pos[0, 0, 0], neg[0, 0, 0] = 0x38, 0xB8            # +1.0 and -1.0
    return oracle.block_scores(pos, w, kb, n, oracle.E4M3)[0] - oracle.block_scores(neg, w, kb, n, oracle.E4M3)[0]


def test_e4m3_widening_spec_values():
    # OCP 8-bit floating point specification, E4M3: bias 7, max normal S.1111.110 = 448,
    # min normal S.0001.000 = 2^-6, max subnormal S.0000.111 = 0.875 x 2^-6, min
    # subnormal S.0000.001 = 2^-9, 1.0 = S.0111.000
    codes = [0x00, 0x80, 0x01, 0x07, 0x08, 0x38, 0x3C, 0x40, 0x7E, 0xFE, 0xB8, 0x81]
    want = [0.0, 0.0, 2.0 ** -9, 0.875 * 2.0 ** -6, 2.0 ** -6, 1.0, 1.5, 2.0, 448.0, -448.0, -1.0, -(2.0 ** -9)]
    np.testing.assert_array_equal(_e4m3_values(codes), want)


def test_e4m3_widening_matches_torch_for_every_finite_code():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)   # 0x7F, 0xFF are NaN
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(_e4m3_values(codes), ref)


def _f16_values(codes):
    """Values of fp16 codes read through the scorer (as _e4m3_values)."""
    kb = np.zeros((len(codes), 128), dtype=np.uint16)
    kb[:, 0] = codes
    n = np.array([len(codes)], np.int32)
    w = np.ones((1, 1), np.float32)
    pos, neg = np.zeros((1, 1, 128), np.uint16), np.zeros((1, 1, 128), np.uint16)
    pos[0, 0, 0], neg[0, 0, 0] = 0x3C00, 0xBC00            # +1.0 and -1.0
    return oracle.block_scores(pos, w, kb, n, oracle.F16)[0] - oracle.block_scores(neg, w, kb, n, oracle.F16)[0]


def test_f16_widening_spec_values():
    # IEEE 754 binary16: bias 15; largest finite 0x7BFF = 65504, smallest normal 0x0400 =
    # 2^-14, smallest subnormal 0x0001 = 2^-24, largest subnormal 0x03FF, 1.0 = 0x3C00
    codes = [0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x3E00, 0x4000, 0x7BFF, 0xFBFF, 0xC000, 0x3555]
    want = [0.0, 0.0, 2.0 ** -24, 1023 * 2.0 ** -24, 2.0 ** -14, 1.0, 1.5, 2.0, 65504.0, -65504.0, -2.0,
            (1024 + 0x155) * 2.0 ** (13 - 25)]
    np.testing.assert_array_equal(_f16_values(codes), want)


def test_f16_widening_matches_numpy_for_every_finite_code():
    codes = np.arange(1 << 16, dtype=np.uint32)
    codes = codes[((codes >> 10) & 0x1F) != 0x1F].astype(np.uint16)      # drop infinities and NaNs
    np.testing.assert_array_equal(_f16_values(codes), codes.view(np.float16).astype(np.float64))


def test_bf16_matches_widened_fp32():
    """Scores of bf16 bits equal the scores of their exact fp32 widening."""
    c = inputs.make_case(21, 2, 4, 30, inputs.BF16, 30 * 64, 8)
    s_bits = oracle.block_scores(c.q, c.w, c.kblk, c.n_blocks, oracle.BF16)
    s_f32 = oracle.block_scores(inputs.bf16_bits_to_f32(c.q), c.w,
                                inputs.bf16_bits_to_f32(c.kblk), c.n_blocks, oracle.F32)
    np.testing.assert_array_equal(s_bits, s_f32)


def test_mask_and_tail_block():
    """Blocks past n are 0; the partial tail block scores like any other block."""
    c = _rand_case(13, nq=2, H=4, C=40)
    full = oracle.block_scores(c.q, c.w, c.kblk, np.array([40, 40], dtype=np.int32))
    n = inputs.blocks_for_tokens([40 * 64 - 63, 17 * 64 + 1])   # 40 and 18 blocks
    np.testing.assert_array_equal(n, [40, 18])
    part = oracle.block_scores(c.q, c.w, c.kblk, n)
    np.testing.assert_array_equal(part[0], full[0])
    np.testing.assert_array_equal(part[1, :18], full[1, :18])
    assert not part[1, 18:].any()
    # the tail block alone, as a one-block context, gives the same score
    one = oracle.block_scores(c.q, c.w, c.kblk[17:18].copy(), np.array([1, 1], dtype=np.int32))
    assert one[1, 0] == full[1, 17]


def test_scores_nonnegative_and_zero_w():
    c = _rand_case(14, nq=2, H=3, C=25)
    s = oracle.block_scores(c.q, c.w, c.kblk, c.n_blocks)
    assert (s >= 0).all()
    z = oracle.block_scores(c.q, np.zeros_like(c.w), c.kblk, c.n_blocks)
    assert not z.any()


# ----------------------------------------------------------------------------- selection

def test_select_hand_fixture(golden_dir):
    g = _load(golden_dir, "select_hand.json")
    for case in g["cases"]:
        sc = np.array(case["scores"], dtype=np.float64)
        n = len(sc)
        row = np.zeros((1, max(n, 1)))
        row[0, :n] = sc
        got = oracle.select(row, np.array([n], dtype=np.int32), case["k"])
        assert got[0].tolist() == case["ids"], case["why"]
        got32 = oracle.select_f32(row.astype(np.float32), np.array([n], dtype=np.int32), case["k"])
        assert got32[0].tolist() == case["ids"], case["why"]


def _brute_force(scores, k):
    """Max-sum k-subset, ties broken by the lexicographically smallest sorted ids."""
    n = len(scores)
    m = min(n, k)
    best = None
    for sub in itertools.combinations(range(n), m):   # generated in lexicographic order
        tot = sum(int(scores[i]) for i in sub)
        if best is None or tot > best[0]:
            best = (tot, sub)
    ids = list(best[1]) if best else []
    return ids + [-1] * (k - m)


def test_select_brute_force_tiny():
    rng = np.random.default_rng(77)
    for trial in range(400):
        n = int(rng.integers(0, 9))
        k = int(rng.integers(1, 7))
        sc = rng.integers(-3, 4, size=n)            # small ints: many ties, exact sums
        row = np.zeros((1, max(n, 1)))
        row[0, :n] = sc
        got = oracle.select(row, np.array([n], dtype=np.int32), k)[0].tolist()
        assert got == _brute_force(sc, k), (sc.tolist(), k, got)


def test_select_closed_forms():
    n, k = 100, 32
    eq = np.full((1, n), 3.5)
    assert oracle.select(eq, np.array([n], np.int32), k)[0].tolist() == list(range(k))
    dec = np.arange(n, 0, -1, dtype=np.float64)[None]
    assert oracle.select(dec, np.array([n], np.int32), k)[0].tolist() == list(range(k))
    inc = np.arange(n, dtype=np.float64)[None]
    assert oracle.select(inc, np.array([n], np.int32), k)[0].tolist() == list(range(n - k, n))
    short = np.arange(10, dtype=np.float64)[None]
    assert oracle.select(short, np.array([10], np.int32), k)[0].tolist() == \
        list(range(10)) + [-1] * (k - 10)
    assert oracle.select(short, np.array([1], np.int32), 4)[0].tolist() == [0, -1, -1, -1]
    assert oracle.select(short, np.array([0], np.int32), 3)[0].tolist() == [-1, -1, -1]


def test_select_64_levels_lowest_ids_on_boundary_level():
    sc = inputs.level_scores(5001, 8, 2048).astype(np.float64)
    k = 32
    n = np.full(8, 2048, dtype=np.int32)
    got = oracle.select(sc, n, k)
    for q in range(8):
        levels = np.unique(sc[q])[::-1]
        above = []
        for lv in levels:                      # walk levels from the top
            ids_at = np.flatnonzero(sc[q] == lv)
            if len(above) + len(ids_at) >= k:
                take = ids_at[: k - len(above)]   # flatnonzero is ascending
                want = sorted(above + take.tolist())
                break
            above += ids_at.tolist()
        assert got[q].tolist() == want


def test_select_invariants_random():
    rng = np.random.default_rng(3)
    for _ in range(50):
        n = int(rng.integers(1, 300))
        k = int(rng.integers(1, 40))
        sc = rng.standard_normal((1, n))
        ids = oracle.select(sc, np.array([n], np.int32), k)[0]
        m = min(n, k)
        sel = ids[:m]
        assert (ids[m:] == -1).all()
        assert (np.diff(sel) > 0).all()                      # ascending, distinct
        rest = np.setdiff1d(np.arange(n), sel)
        if len(rest):
            assert sc[0, sel].min() >= sc[0, rest].max()


def test_clamping_of_n_blocks():
    sc = np.arange(8, dtype=np.float64)[None]
    assert oracle.select(sc, np.array([50], np.int32), 3)[0].tolist() == [5, 6, 7]
    assert oracle.select(sc, np.array([-4], np.int32), 2)[0].tolist() == [-1, -1]


# ----------------------------------------------------------------------------- mutation

MUTANTS = {
    "relu_dropped": ("double relu = dot > 0.0 ? dot : 0.0;\n                    s += (double)w[(size_t)qi * n_heads + h] * relu;",
                       "s += (double)w[(size_t)qi * n_heads + h] * dot;"),
    "tie_to_higher_id": ("return (a->id > b->id) - (a->id < b->id);",
                         "return (a->id < b->id) - (a->id > b->id);"),
    "ascending_scores": ("if (a->score > b->score) return -1;", "if (a->score < b->score) return -2;"),
    "unsorted_emit": ("qsort(out, (size_t)m, sizeof *out, by_int_asc);", ""),
    "transposed_q_index": ("size_t qrow = ((size_t)qi * n_heads + h) * head_dim;",
                           "size_t qrow = ((size_t)h * nq + qi) * head_dim;"),
    "dropped_last_d": ("for (int d = 0; d < head_dim; ++d)", "for (int d = 0; d + 1 < head_dim; ++d)"),
    "w_wrong_head": ("s += (double)w[(size_t)qi * n_heads + h] * relu;",
                     "s += (double)w[(size_t)qi * n_heads] * relu;"),
    "bf16_wrong_shift": ("uint32_t u = ((uint32_t)h) << 16;", "uint32_t u = ((uint32_t)h) << 15;"),
    "no_pad": ("for (int i = m; i < k; ++i) out[i] = -1;", "for (int i = m; i < k; ++i) out[i] = 0;"),
    "e4m3_bias": ("v = ldexp(8.0 + m, e - 10);", "v = ldexp(8.0 + m, e - 9);"),
    "e4m3_subnormal": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "e4m3_sign": ("return (b & 0x80) ? -v : v;", "return v;"),
    "f16_bias": ("v = ldexp(1024.0 + m, e - 25);", "v = ldexp(1024.0 + m, e - 24);"),
    "f16_subnormal": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "f16_sign": ("return (b & 0x8000) ? -v : v;", "return v;"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_pins_catch_planted_oracle_mistakes(tmp_path, golden_dir, monkeypatch):
    """Compile mutated copies of the oracle; the pins above must fail on each one."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "qsa_oracle.c")).read()
    pins = [test_scores_hand_fixture, test_bf16_widening_fixture, test_relu_per_head_identities,
            test_exactly_rounded_sum_crosscheck, test_select_hand_fixture,
            test_select_brute_force_tiny, test_select_closed_forms,
            test_select_64_levels_lowest_ids_on_boundary_level, test_e4m3_widening_spec_values,
            test_f16_widening_spec_values]
    for name, (old, new) in MUTANTS.items():
        assert old in src, name
        msrc = tmp_path / f"{name}.c"
        msrc.write_text(src.replace(old, new, 1))
        so = tmp_path / f"{name}.so"
        subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-w", "-o", str(so), str(msrc), "-lm"], check=True)
        monkeypatch.setattr(oracle, "_lib", None)
        monkeypatch.setattr(oracle, "_LIB", str(so))
        monkeypatch.setattr(oracle, "build", lambda force=False: str(so))
        caught = False
        for pin in pins:
            args = [golden_dir] if pin.__code__.co_argcount else []
            try:
                pin(*args)
            except AssertionError:
                caught = True
                break
        monkeypatch.setattr(oracle, "_lib", None)
        assert caught, f"no pin caught the planted mistake '{name}'"
