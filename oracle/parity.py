"""Parity rules between the CUDA path's outputs and the oracle's (test
infrastructure, like the rest of this package: used by the GPU tests, the smoke
check and the benchmark's parity report, outside any timed region).

Rule (a): the GPU's top-k ids equal the oracle's selection over the GPU's own
          fp32 scores, bit for bit.
Rule (b): per query, max_b |gpu - ref| / max_b |ref| <= tol (ref = FP64 oracle
          scores; tol 1e-4 for fp32 and fp8 e4m3 inputs, 1e-2 for bf16).  A query whose
          reference scale is 0 must give exactly 0.
Rule (c): the end-to-end ids equal the oracle's FP64 selection, except for a
          query whose FP64 gap at the k-th boundary, (s_(k) - s_(k+1)) / scale,
          is below tol; such a query is counted and must still be a valid
          tolerance top-k (every selected ref >= s_(k) - tol*scale, every other
          ref <= s_(k) + tol*scale).  Exact FP64 ties (gap 0) are not excused.
Rule (d), selection attention: per (query, head, dim),
          |o_gpu - o_ref| <= (2u + 2^-12) * sum_t w_t |v_t| + a, and
          |lse_gpu - lse_ref| <= u + 1e-5 (1 + |lse_ref|), with u the unit
          roundoff of the weights' format (2^-9 bf16, 2^-11 fp16).  The GPU
          rounds each weight to that format and divides by the sum of the
          rounded weights, so every normalised weight is within 2u (1 + u) of
          the exact one; 2^-12 covers the fp32 accumulation.  a = 1e-7, plus for
          fp16 the weights that fall below its normal range (absolute error at
          most 2^-25 each, at most 64 k of them, the largest weight being 1):
          64 k 2^-25 max|V|.  sum_t w_t |v_t| is the oracle's output on |V|.  An
          empty token set gives exactly 0 and -inf.
"""
from __future__ import annotations

import numpy as np

# Tolerance of rules (b) and (c) by dtype code.  fp32 and bf16: the values the
# selection path's specification fixes.  fp8 e4m3 (keys and queries stored in 8
# bits): every product of two e4m3 values is exact in fp32 (4-bit significands, so
# 8-bit products, exponents far inside fp32's range), and the 128 products and the
# head-weighted sum accumulate in fp32, so the scorer rounds like the fp32 path:
# the fp32 tolerance applies.  Measured: 1.3e-7 at most (decode and deep prompt).
TOL = {0: 1e-4, 1: 1e-2, 2: 1e-4}   # fp32, bf16, fp8 e4m3


def score_errors(gpu: np.ndarray, ref: np.ndarray, n_blocks: np.ndarray) -> np.ndarray:
    """Per-query max |gpu - ref| / max |ref| over the valid blocks (0 if none)."""
    out = np.zeros(len(n_blocks))
    for q, n in enumerate(n_blocks):
        n = int(n)
        if n == 0:
            continue
        scale = np.abs(ref[q, :n]).max()
        err = np.abs(gpu[q, :n].astype(np.float64) - ref[q, :n]).max()
        out[q] = err / scale if scale > 0 else (0.0 if err == 0 else np.inf)
    return out


def check_rule_b(gpu, ref, n_blocks, dtype):
    e = score_errors(gpu, ref, n_blocks)
    assert np.isfinite(e).all(), "a zero-scale query gave a nonzero score"
    assert e.max() <= TOL[dtype], f"rule (b): max normalised score error {e.max():.3e} > {TOL[dtype]}"
    return float(e.max())


def check_rule_a(gpu_ids, oracle_ids_on_gpu_scores):
    bad = np.flatnonzero((gpu_ids != oracle_ids_on_gpu_scores).any(1))
    assert len(bad) == 0, f"rule (a): {len(bad)} queries differ, first {bad[:5].tolist()}: " \
        f"gpu {gpu_ids[bad[0]].tolist()} oracle {oracle_ids_on_gpu_scores[bad[0]].tolist()}"


def rule_c(gpu_ids, ref_scores, ref_ids, n_blocks, k, tol, tight_tol=None):
    """Counts: exact, excused (near-tie, valid), failed; and near-ties at tight_tol."""
    res = {"queries": len(n_blocks), "exact": 0, "excused": 0, "failed": 0, "near_tie": 0,
           "near_tie_tight": 0, "failed_ids": []}
    for q, n in enumerate(n_blocks):
        n = int(n)
        same = (gpu_ids[q] == ref_ids[q]).all()
        if n <= k:
            res["exact" if same else "failed"] += 1
            if not same:
                res["failed_ids"].append(q)
            continue
        row = ref_scores[q, :n]
        scale = np.abs(row).max()
        srt = np.sort(row)[::-1]
        sk, sk1 = srt[k - 1], srt[k]
        gap = (sk - sk1) / scale if scale > 0 else 0.0
        if gap < tol and gap > 0:
            res["near_tie"] += 1
        if tight_tol is not None and gap < tight_tol and gap > 0:
            res["near_tie_tight"] += 1
        if same:
            res["exact"] += 1
            continue
        sel = gpu_ids[q][gpu_ids[q] >= 0]
        valid = len(sel) == k and len(np.unique(sel)) == k and (np.diff(sel) > 0).all() and sel.max() < n
        if valid and gap > 0 and gap < tol:
            mask = np.zeros(n, bool)
            mask[sel] = True
            ok = row[mask].min() >= sk - tol * scale and (not (~mask).any() or
                                                         row[~mask].max() <= sk + tol * scale)
            if ok:
                res["excused"] += 1
                continue
        res["failed"] += 1
        res["failed_ids"].append(q)
    return res


def check_rule_c(gpu_ids, ref_scores, ref_ids, n_blocks, k, dtype, tight_tol=None):
    r = rule_c(gpu_ids, ref_scores, ref_ids, n_blocks, k, TOL[dtype], tight_tol)
    assert r["failed"] == 0, f"rule (c): {r['failed']} queries fail, first {r['failed_ids'][:5]}"
    return r


ATTN_U = {1: 2.0 ** -9, 3: 2.0 ** -11}   # unit roundoff of the weights: bf16, fp16


def attention_reference(case, rows=None):
    """Oracle (out, lse, bounds) for the queries ``rows`` (all by default); bounds is what
    check_rule_d needs: sum_t w_t |v_t| (the oracle's output on |V|), the weights'
    unit roundoff and the absolute term."""
    import oracle
    r = slice(None) if rows is None else np.asarray(rows)
    qa, ids, nt = case.qa[r], case.ids[r], case.n_tokens[r]
    out, lse = oracle.select_attention(qa, case.kc, case.vc, ids, nt, case.scale, case.dtype)
    wabs, _ = oracle.select_attention(qa, case.kc, case.vc & np.uint16(0x7FFF), ids, nt, case.scale, case.dtype)
    u = ATTN_U[case.dtype]
    extra = 1e-7
    if case.dtype == oracle.F16:
        v = np.abs(case.vc.view(np.float16).astype(np.float32))
        vmax = float(v[np.isfinite(v)].max())   # rows past a context may hold anything
        extra += 64 * case.k * 2.0 ** -25 * vmax
    return out, lse, (wabs, u, extra)


def check_rule_d(out_gpu, lse_gpu, out_ref, lse_ref, bounds):
    """Assert rule (d); returns the largest error as a fraction of its bound."""
    wabs, u, extra = bounds
    out_gpu = np.asarray(out_gpu, np.float64)
    empty = np.isneginf(lse_ref)
    assert (out_gpu[empty] == 0).all(), "an empty token set gave a nonzero output"
    if lse_gpu is not None:
        assert np.isneginf(np.asarray(lse_gpu)[empty]).all(), "an empty token set gave a finite lse"
    full = ~empty
    bound = (2 * u + 2.0 ** -12) * wabs[full] + extra
    err = np.abs(out_gpu[full] - out_ref[full])
    assert np.isfinite(out_gpu[full]).all(), "non-finite output"
    worst = float((err / bound).max()) if err.size else 0.0
    assert worst <= 1.0, f"rule (d): output error {worst:.3f} x its bound"
    if lse_gpu is not None and full.any():
        lg = np.asarray(lse_gpu, np.float64)[full]
        lb = u + 1e-5 * (1 + np.abs(lse_ref[full]))
        le = np.abs(lg - lse_ref[full])
        assert (le <= lb).all(), f"rule (d): lse error {float((le / lb).max()):.3f} x its bound"
        worst = max(worst, float((le / lb).max()))
    return worst
