"""The seeded input generator: bf16 and e4m3 rounding, block counts, determinism."""
import numpy as np
import pytest

from workloads import inputs


def test_bf16_rounding_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 3.140625, 0.0],
                 dtype=np.float32)
    bits = inputs.to_bf16_bits(x)
    # 1 + 2^-8 is half way between 1 and 1 + 2^-7: ties to even -> 1.0;
    # 1 + 3*2^-8 is half way between 1 + 2^-7 and 1 + 2^-6: ties to even -> 1 + 2^-6
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0x3F80, 0xC020, 0x4049, 0x0000]
    back = inputs.bf16_bits_to_f32(bits)
    assert back.tolist() == [1.0, 1.0, 1.0 + 2**-6, 1.0, -2.5, 3.140625, 0.0]


def test_bf16_roundtrip_exact_on_bf16_values():
    rng = np.random.default_rng(0)
    b = rng.integers(0, 2**16, size=4096, dtype=np.uint16)
    f = inputs.bf16_bits_to_f32(b)
    ok = np.isfinite(f)
    assert (inputs.to_bf16_bits(f[ok]) == b[ok]).all()


def test_blocks_for_tokens():
    assert inputs.blocks_for_tokens([1, 63, 64, 65, 4096, 40_000, 40_001, 258_000, 520_000,
                                     131_072]).tolist() == \
        [1, 1, 1, 2, 64, 625, 626, 4032, 8125, 2048]


def test_named_workloads_shapes_and_determinism():
    t = inputs.tiny_case()
    assert t.q.shape == (1, 8, 128) and t.q.dtype == np.float32 and t.n_blocks.tolist() == [64]
    d = inputs.decode_case(5)
    assert d.q.shape == (3, 16, 128) and d.q.dtype == np.uint16 and d.max_blocks == 4096
    assert d.n_blocks.tolist() == [4032] * 3 and d.k == 32 and d.active_blocks == -1
    a = inputs.deep_case(2)
    assert a.n_blocks[0] == 8125 and a.max_blocks == 8192 and a.active_blocks == 8125
    b = inputs.deep_case(2)
    assert (a.q == b.q).all() and (a.kblk == b.kblk).all() and (a.w == b.w).all()
    r = inputs.stress_case("ragged")
    assert r.n_blocks.min() >= 1 and r.n_blocks.max() <= 2048
    assert (r.tokens % 64 != 0).any()


def test_e4m3_rounding_matches_torch_and_breaks_ties_to_even():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * s for s in (1e-3, 1.0, 30.0)])
    mids = ((inputs._E4M3_VALUES[:-1] + inputs._E4M3_VALUES[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, np.float32([0.0, -0.0, 448.0, -448.0])])
    ours = inputs.to_e4m3_bits(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)
    assert inputs.to_e4m3_bits(np.float32([1e6, -1e6])).tolist() == [0x7E, 0xFE]   # saturated


def test_parallel_normal_draws_do_not_depend_on_the_thread_count(monkeypatch):
    import os
    a = inputs.normal_16bit(11, (3, 1000, 128))
    monkeypatch.setattr(os, "cpu_count", lambda: 1)     # one worker fills every slice in turn
    b = inputs.normal_16bit(11, (3, 1000, 128))
    np.testing.assert_array_equal(a, b)
    c = inputs.normal_16bit(11, (3, 1000, 128), dtype=inputs.F16)
    assert np.isfinite(c.view(np.float16)).all() and not np.array_equal(c, a)
