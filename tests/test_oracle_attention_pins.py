"""Pins of the selection-attention oracle against facts fixed outside it.

Closed forms worked by hand (two tokens, one token, equal keys), a library
routine on the special case "every block selected" (dense causal attention,
torch's scaled_dot_product_attention in float64), invariances of the token set
(slot order, pads, duplicates), the GQA head-to-KV-head map read off constant
values, overflow safety, the causal tail, and empty sets.  A mutation test
plants plausible mistakes in a copy of the oracle and checks that the pins
catch every one.
"""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from workloads import inputs

bf16 = inputs.to_bf16_bits


def _bits(x, dtype):
    x = np.asarray(x, np.float32)
    return inputs.to_f16_bits(x) if dtype == oracle.F16 else bf16(x)


def _attn(qa, kc, vc, ids, n_tokens, scale, dtype=oracle.BF16):
    return oracle.select_attention(_bits(qa, dtype), _bits(kc, dtype), _bits(vc, dtype), np.asarray(ids, np.int32),
                                   np.asarray(n_tokens, np.int32), scale, dtype)


def test_two_tokens_closed_form(dtype=oracle.BF16):
    # block 1 of a 66-token context holds tokens 64 and 65; every other row would
    # dominate (or stand out) if it leaked in
    kc = np.full((1, 128, 2), 8.0, np.float32)
    vc = np.full((1, 128, 2), 100.0, np.float32)
    vc[0, :, 1] = -100.0
    kc[0, 64], kc[0, 65] = (1.0, 0.0), (0.0, 1.0)
    vc[0, 64], vc[0, 65] = (1.0, 2.0), (3.0, 4.0)
    qa = np.array([[[1.0, 0.0], [0.0, 2.0]]], np.float32)
    out, lse = _attn(qa, kc, vc, [[1, -1]], [66], 0.5, dtype)
    e = math.exp(0.5)
    a0, b0 = e / (e + 1), 1 / (e + 1)                       # head 0: logits 0.5, 0
    a1, b1 = 1 / (1 + math.e), math.e / (1 + math.e)        # head 1: logits 0, 1
    np.testing.assert_allclose(out[0, 0], [a0 + 3 * b0, 2 * a0 + 4 * b0], rtol=1e-14)
    np.testing.assert_allclose(out[0, 1], [a1 + 3 * b1, 2 * a1 + 4 * b1], rtol=1e-14)
    np.testing.assert_allclose(lse[0], [math.log(e + 1), math.log(1 + math.e)], rtol=1e-14)


def test_single_token_is_its_value():
    c = inputs.make_attention_case(71, 4, 2, 512, 512, 4)
    b = np.array([3, 0, 7, 5])
    n_tokens = b * 64 + 1                     # only the first token of block b is visible
    ids = np.full((4, 4), -1, np.int32)
    ids[:, 0] = b
    out, lse = oracle.select_attention(c.qa, c.kc, c.vc, ids, n_tokens, c.scale)
    v = inputs.bf16_bits_to_f32(c.vc).astype(np.float64)
    for q in range(4):
        for h in range(c.n_heads):
            np.testing.assert_array_equal(out[q, h], v[h // 16, 64 * b[q]])
    assert np.isfinite(lse).all()


def test_equal_keys_give_the_mean_of_values():
    c = inputs.make_attention_case(72, 2, 1, 256, [256, 150], 4)
    kc = c.kc.copy()
    kc[:] = kc[0, 0]
    qa = c.qa.copy()
    qa[1] = qa[0]                            # one query vector, two token sets
    ids = np.array([[0, 2, 3, -1], [1, 2, -1, -1]], np.int32)
    out, lse = oracle.select_attention(qa, kc, c.vc, ids, c.n_tokens, c.scale)
    v = inputs.bf16_bits_to_f32(c.vc).astype(np.float64)[0]
    for q, toks in enumerate([np.r_[0:64, 128:256], np.r_[64:150]]):
        want = np.array([math.fsum(v[toks, d]) / len(toks) for d in range(128)])
        for h in range(c.n_heads):
            np.testing.assert_allclose(out[q, h], want, rtol=1e-12, atol=1e-13)
        assert np.ptp(lse[q]) > 0            # heads differ
    # every logit of a head is the same s: lse = s + log(n)
    assert (np.abs(lse[0] - lse[1] - (math.log(192) - math.log(86))) < 1e-12).all()


def test_every_block_selected_is_dense_causal_attention(dtype=oracle.BF16):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    n_tokens = [300, 64, 257, 1]
    c = inputs.make_attention_case(73, 4, 2, 320, n_tokens, 5, group=3, dtype=dtype)
    nb = inputs.blocks_for_tokens(c.n_tokens)
    ids = np.full((4, 5), -1, np.int32)
    for q in range(4):
        ids[q, :nb[q]] = np.arange(nb[q])
    out, lse = oracle.select_attention(c.qa, c.kc, c.vc, ids, c.n_tokens, c.scale, dtype)
    qf = torch.from_numpy(inputs.bits_to_f32(c.qa, dtype).astype(np.float64))
    kf = torch.from_numpy(inputs.bits_to_f32(c.kc, dtype).astype(np.float64))
    vf = torch.from_numpy(inputs.bits_to_f32(c.vc, dtype).astype(np.float64))
    for q in range(4):
        n = n_tokens[q]
        for h in range(c.n_heads):
            g = h // 3
            ref = F.scaled_dot_product_attention(qf[q, h][None, None], kf[g, :n][None], vf[g, :n][None],
                                                 scale=c.scale)[0, 0]
            np.testing.assert_allclose(out[q, h], ref.numpy(), rtol=1e-11, atol=1e-12)
            ref_lse = torch.logsumexp(c.scale * (kf[g, :n] @ qf[q, h]), 0).item()
            assert abs(lse[q, h] - ref_lse) < 1e-11


def test_two_tokens_closed_form_f16():
    test_two_tokens_closed_form(oracle.F16)


def test_every_block_selected_is_dense_causal_attention_f16():
    test_every_block_selected_is_dense_causal_attention(oracle.F16)


def test_slot_order_pads_and_duplicates_do_not_matter():
    c = inputs.make_attention_case(74, 3, 1, 1024, [1024, 700, 1000], 6)
    out, lse = oracle.select_attention(c.qa, c.kc, c.vc, c.ids, c.n_tokens, c.scale)
    rng = np.random.default_rng(0)
    mixed = np.full((3, 10), -1, np.int32)
    for q in range(3):
        row = [int(b) for b in c.ids[q] if b >= 0]
        row = row + [row[0], row[-1]]          # duplicates
        slots = rng.permutation(10)[:len(row)]
        mixed[q, slots] = rng.permutation(row)
    out2, lse2 = oracle.select_attention(c.qa, c.kc, c.vc, mixed, c.n_tokens, c.scale)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)


def test_gqa_heads_read_their_group_kv_head():
    c = inputs.make_attention_case(75, 2, 3, 256, 256, 3, group=4)
    vc = np.empty_like(c.vc)
    for g in range(3):   # powers of two: the weighted mean of a constant is exact
        vc[g] = bf16(np.full((256, 128), 2.0 ** g, np.float32))
    out, _ = oracle.select_attention(c.qa, c.kc, vc, c.ids, c.n_tokens, c.scale)
    for h in range(12):
        assert (out[:, h] == 2.0 ** (h // 4)).all()


def test_large_logits_stay_finite():
    c = inputs.make_attention_case(76, 2, 1, 512, 512, 8)
    qa = bf16(inputs.bf16_bits_to_f32(c.qa) * 256.0)     # logits in the thousands
    out, lse = oracle.select_attention(qa, c.kc, c.vc, c.ids, c.n_tokens, c.scale)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    v = inputs.bf16_bits_to_f32(c.vc).astype(np.float64)[0]
    # a convex combination of the value rows: inside their per-dimension range
    assert (out <= v.max(axis=0) + 1e-12).all() and (out >= v.min(axis=0) - 1e-12).all()
    assert (lse > 100).all()


def test_tokens_at_or_past_the_context_are_excluded():
    c = inputs.make_attention_case(77, 1, 1, 512, 64 * 5 + 17, 3)
    ids = np.array([[1, 5, -1]], np.int32)
    out, lse = oracle.select_attention(c.qa, c.kc, c.vc, ids, c.n_tokens, c.scale)
    kc, vc = c.kc.copy(), c.vc.copy()
    kc[0, 64 * 5 + 17:] = bf16(np.full(128, 30.0, np.float32))   # would dominate if visible
    vc[0, 64 * 5 + 17:] = bf16(np.full(128, 7.0, np.float32))
    out2, lse2 = oracle.select_attention(c.qa, kc, vc, ids, c.n_tokens, c.scale)
    np.testing.assert_array_equal(out2, out)
    np.testing.assert_array_equal(lse2, lse)
    vc[0, 64 * 5 + 16] = bf16(np.full(128, 7.0, np.float32))     # the last visible token counts
    out3, _ = oracle.select_attention(c.qa, kc, vc, ids, c.n_tokens, c.scale)
    assert (np.abs(out3 - out) > 0).any()


def test_empty_token_sets():
    c = inputs.make_attention_case(78, 4, 1, 256, [256, 0, 100, 256], 2)
    ids = np.array([[-1, -1], [0, 1], [2, 3], [-1, -1]], np.int32)   # pads; no context; past the context
    out, lse = oracle.select_attention(c.qa, c.kc, c.vc, ids, c.n_tokens, c.scale)
    assert (out == 0).all()
    assert np.isneginf(lse).all()


# ----------------------------------------------------------------------------- mutation

PINS = [test_two_tokens_closed_form, test_single_token_is_its_value, test_equal_keys_give_the_mean_of_values,
        test_every_block_selected_is_dense_causal_attention, test_slot_order_pads_and_duplicates_do_not_matter,
        test_gqa_heads_read_their_group_kv_head, test_large_logits_stay_finite,
        test_tokens_at_or_past_the_context_are_excluded, test_empty_token_sets]

MUTANTS = {
    "scale_dropped": ("s[i] = scale * dot;", "s[i] = dot;"),
    "group_by_modulo": ("const int g = h / group;", "const int g = h % n_kv_heads;"),
    "tail_inclusive": ("if (t < ntok) tok[n++] = (int32_t)t;", "if (t <= ntok && t < capacity) tok[n++] = (int32_t)t;"),
    "no_max_shift": ("const double e = exp(s[i] - m);", "const double e = exp(s[i]);"),
    "lse_without_max": ("lse[(size_t)qi * n_heads + h] = m + log(l);", "lse[(size_t)qi * n_heads + h] = log(l);"),
    "no_dedup": ("if (seen) continue;", ""),
    "values_from_keys": ("o[d] += e * widen(vc, dtype, vrow + d);", "o[d] += e * widen(kc, dtype, vrow + d);"),
    "transposed_q_index": ("const size_t qrow = ((size_t)qi * n_heads + h) * head_dim;",
                           "const size_t qrow = ((size_t)h * nq + qi) * head_dim;"),
    "no_normalise": ("for (int d = 0; d < head_dim; ++d) o[d] /= l;", ""),
    "block_stride_off": ("const int64_t t = (int64_t)b * 64 + r;", "const int64_t t = (int64_t)b * 63 + r;"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_pins_catch_planted_attention_mistakes(tmp_path, monkeypatch):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "qsa_oracle.c")).read()
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
        for pin in PINS:
            try:
                with np.errstate(all="ignore"):
                    pin()
            except AssertionError:
                caught = True
                break
        monkeypatch.setattr(oracle, "_lib", None)
        assert caught, f"no pin caught the planted mistake '{name}'"
