"""Seeded synthetic inputs for block selection, shared by the tests, the smoke
check and the benchmark.

This module holds no arithmetic of the method: it only draws random arrays
(numpy PCG64), rounds them to bf16 storage, and names the workload shapes.
Both the CUDA path and the CPU oracle are fed from here.

Workloads (synthetic stand-ins for the pages' bench data: queries, indexer
heads and keys drawn i.i.d., one key per 64-token KV block, the last block
partial when the context is not a multiple of 64):

* ``tiny``   -- 1 query, 8 heads, fp32, 4,096 tokens (64 blocks), k = 16
* ``decode`` -- 3 queries, 16 heads, bf16, capacity 262,144 tokens (4,096 blocks),
  contexts 40K/64K/131K/258K tokens (+ 40,001 and 64,001), k = 32, no active count
* ``prompt`` -- 256 queries, 16 heads, bf16, 131,072 tokens (2,048 blocks), k = 32
* ``deep``   -- 256 queries, 16 heads, bf16, capacity 524,288 tokens (8,192 blocks),
  contexts 262K/400K/520K tokens (up to 8,125 blocks), k = 32
* ``stress`` -- 256 queries at 131,072 tokens: all-equal scores, 64-level scores,
  w = 0, and per-query contexts of 1..2,048 blocks with a partial tail.

"K" in a context size is decimal (520K = 520,000 tokens = 8,125 blocks), except
131,072, which is written out.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK_TOKENS = 64
HEAD_DIM = 128
F32 = 0
BF16 = 1
E4M3 = 2


def blocks_for_tokens(tokens):
    """Number of 64-token blocks covering ``tokens`` tokens (last one partial)."""
    t = np.asarray(tokens, dtype=np.int64)
    return ((t + BLOCK_TOKENS - 1) // BLOCK_TOKENS).astype(np.int32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (inputs are finite:
    the largest finite pattern plus the rounding increment stays below 2^32)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).reshape(-1)
    out = np.empty(u.shape, dtype=np.uint16)
    step = 1 << 24
    for i in range(0, u.size, step):   # bounded temporaries on large caches
        c = u[i:i + step]
        out[i:i + step] = (c + np.uint32(0x7FFF) + ((c >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return out.reshape(np.shape(x))


def _e4m3_codes_values():
    """Values of the non-negative finite e4m3 codes 0x00 .. 0x7E (ascending): OCP 8-bit
    floating point E4M3, bias 7, exponent 0 holding the subnormals."""
    codes = np.arange(0x7F, dtype=np.int64)
    e, m = (codes >> 3) & 0xF, codes & 7
    return np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e - 10.0))


_E4M3_VALUES = _e4m3_codes_values()
_E4M3_MIDS = (_E4M3_VALUES[:-1] + _E4M3_VALUES[1:]) / 2


def to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> e4m3 bit patterns (uint8): nearest value, ties to the even code,
    magnitudes past 448 saturated to 448 (inputs are finite)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64).reshape(-1)
    idx = np.searchsorted(_E4M3_MIDS, a, side="left")       # ties land on the lower code
    tie = (idx < len(_E4M3_MIDS)) & (a == _E4M3_MIDS[np.minimum(idx, len(_E4M3_MIDS) - 1)])
    idx = np.where(tie & (idx % 2 == 1), idx + 1, idx)
    idx = np.minimum(idx, 0x7E)
    sign = np.signbit(x).reshape(-1).astype(np.uint8) << 7
    return (idx.astype(np.uint8) | sign).reshape(x.shape)


F16 = 3


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> IEEE binary16 bit patterns (uint16), round to nearest even (numpy's cast)."""
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32).astype(np.float16)).view(np.uint16)


def bits_to_f32(bits: np.ndarray, dtype: int) -> np.ndarray:
    """bf16 or fp16 bit patterns (uint16) -> fp32 values (exact)."""
    if dtype == F16:
        return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)
    return bf16_bits_to_f32(bits)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Case:
    """One synthetic selection problem.

    ``q`` [nq,H,D] and ``kblk`` [C,D] hold fp32 values (dtype F32), bf16 bit
    patterns as uint16 (dtype BF16) or fp8 e4m3 bit patterns as uint8 (dtype E4M3); ``w`` [nq,H] is fp32; ``n_blocks`` [nq]
    int32.  ``tokens`` is the per-query context length the blocks cover.
    """
    q: np.ndarray
    w: np.ndarray
    kblk: np.ndarray
    n_blocks: np.ndarray
    tokens: np.ndarray
    dtype: int
    k: int
    active_blocks: int = -1
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def nq(self) -> int:
        return self.q.shape[0]

    @property
    def n_heads(self) -> int:
        return self.q.shape[1]

    @property
    def max_blocks(self) -> int:
        return self.kblk.shape[0]


def make_case(seed: int, nq: int, n_heads: int, capacity_blocks: int, dtype: int,
              tokens, k: int, *, active_blocks: int = -1, w_zero: bool = False,
              kblk_equal: bool = False, name: str = "") -> Case:
    """q, kblk ~ N(0,1), w ~ U(0,1) from ``seed``; ``tokens`` scalar or per query.

    Rows of kblk at or past a query's block count are random too, so masking
    is exercised.  bf16 storage rounds the fp32 draws to nearest even.
    """
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((nq, n_heads, HEAD_DIM), dtype=np.float32)
    kblk = rng.standard_normal((capacity_blocks, HEAD_DIM), dtype=np.float32)
    w = rng.random((nq, n_heads), dtype=np.float32)
    if w_zero:
        w[:] = 0.0
    if kblk_equal:
        kblk[:] = kblk[0]
    toks = np.broadcast_to(np.asarray(tokens, dtype=np.int64), (nq,)).copy()
    n_blocks = blocks_for_tokens(toks)
    if dtype == BF16:
        q = to_bf16_bits(q)
        kblk = to_bf16_bits(kblk)
    elif dtype == E4M3:
        q = to_e4m3_bits(q)
        kblk = to_e4m3_bits(kblk)
    return Case(q=q, w=w, kblk=kblk, n_blocks=n_blocks, tokens=toks, dtype=dtype, k=k,
                active_blocks=active_blocks, name=name)


def ragged_tokens(seed: int, nq: int, max_full_blocks: int) -> np.ndarray:
    """Per-query contexts of U{1..max_full_blocks} blocks, the last one holding U{1..64} tokens."""
    rng = np.random.default_rng(seed)
    nb = rng.integers(1, max_full_blocks + 1, size=nq)
    tail = rng.integers(1, BLOCK_TOKENS + 1, size=nq)
    return (nb - 1) * BLOCK_TOKENS + tail


def level_scores(seed: int, nq: int, cols: int, levels: int = 64) -> np.ndarray:
    """Scores quantised to ``levels`` levels: floor(U * levels) / levels, fp32."""
    rng = np.random.default_rng(seed)
    u = rng.random((nq, cols))
    return (np.floor(u * levels) / levels).astype(np.float32)


def normal_scores(seed: int, nq: int, cols: int) -> np.ndarray:
    """Continuous scores ~ N(0,1), fp32 (negative values included)."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((nq, cols), dtype=np.float32)


# Named workloads: seed = 1000 * config index + sweep index.
DECODE_TOKENS = (40_000, 40_001, 64_000, 64_001, 131_000, 258_000)
DEEP_TOKENS = (262_000, 400_000, 520_000)


def tiny_case() -> Case:
    return make_case(1000, 1, 8, 64, F32, 4096, 16, name="tiny 1q x 8h fp32, 4,096 tokens")


def decode_case(i: int) -> Case:
    t = DECODE_TOKENS[i]
    return make_case(2000 + i, 3, 16, 4096, BF16, t, 32,
                     name=f"decode 3q x 16h bf16, {t:,} tokens, capacity 262,144")


def prompt_case() -> Case:
    return make_case(3000, 256, 16, 2048, BF16, 131_072, 32, active_blocks=2048,
                     name="prompt 256q x 16h bf16, 131,072 tokens")


def deep_case(i: int) -> Case:
    t = DEEP_TOKENS[i]
    nb = int(blocks_for_tokens(t))
    return make_case(4000 + i, 256, 16, 8192, BF16, t, 32, active_blocks=nb,
                     name=f"deep 256q x 16h bf16, {t:,} tokens, capacity 524,288")


def deep_e4m3_case() -> Case:
    """The deep prompt at 520,000 tokens with q and kblk stored as fp8 e4m3 (the same
    N(0,1) draws as the bf16 case, rounded to e4m3)."""
    return make_case(4002, 256, 16, 8192, E4M3, 520_000, 32, active_blocks=8125,
                     name="deep 256q x 16h e4m3, 520,000 tokens, capacity 524,288")


def decode_e4m3_case() -> Case:
    return make_case(2005, 3, 16, 4096, E4M3, 258_000, 32,
                     name="decode 3q x 16h e4m3, 258,000 tokens, capacity 262,144")


def stress_case(kind: str) -> Case:
    """End-to-end stress cases at 256 queries and 131,072 tokens."""
    if kind == "equal_kblk":
        return make_case(5000, 256, 16, 2048, BF16, 131_072, 32, active_blocks=2048,
                         kblk_equal=True, name="stress: every kblk row identical")
    if kind == "w_zero":
        return make_case(5002, 256, 16, 2048, BF16, 131_072, 32, active_blocks=2048,
                         w_zero=True, name="stress: w = 0")
    if kind == "ragged":
        toks = ragged_tokens(5003, 256, 2048)
        return make_case(5003, 256, 16, 2048, BF16, toks, 32, active_blocks=2048,
                         name="stress: per-query contexts 1..2,048 blocks, partial tail")
    raise ValueError(kind)


# ----------------------------------------------------------------------------- selection attention

@dataclass
class AttnCase:
    """One synthetic selection-attention problem.

    ``qa`` [nq,H,128] and ``kc``/``vc`` [Hkv,C,128] (token rows) hold bf16 bit
    patterns (uint16) drawn N(0,1); ``ids`` [nq,k] int32 are distinct block ids
    inside each query's context, ascending, -1 padded; ``n_tokens`` [nq] int32.
    The heads of a GQA group (``H / Hkv`` of them) share one KV head.
    """
    qa: np.ndarray
    kc: np.ndarray
    vc: np.ndarray
    ids: np.ndarray
    n_tokens: np.ndarray
    scale: float
    name: str = ""
    dtype: int = BF16                   # BF16 or F16: the bit patterns' format

    @property
    def nq(self) -> int:
        return self.qa.shape[0]

    @property
    def n_heads(self) -> int:
        return self.qa.shape[1]

    @property
    def n_kv_heads(self) -> int:
        return self.kc.shape[0]

    @property
    def capacity(self) -> int:
        return self.kc.shape[1]

    @property
    def k(self) -> int:
        return self.ids.shape[1]


def random_ids(seed: int, n_blocks, k: int, n_valid=None) -> np.ndarray:
    """Per query, min(n_valid, n_blocks, k) distinct ids drawn uniformly from
    [0, n_blocks), ascending, then -1 (the path's output format)."""
    rng = np.random.default_rng(seed)
    nb = np.asarray(n_blocks, dtype=np.int64)
    nv = nb if n_valid is None else np.minimum(np.asarray(n_valid, dtype=np.int64), nb)
    out = np.full((len(nb), k), -1, dtype=np.int32)
    for i, (n, v) in enumerate(zip(nb, nv)):
        m = int(min(v, k))
        if m > 0:
            out[i, :m] = np.sort(rng.choice(int(n), size=m, replace=False))
    return out


def normal_16bit(seed: int, shape, chunks: int = 16, dtype: int = BF16) -> np.ndarray:
    """N(0,1) draws rounded to bf16 (or fp16) bits, in ``chunks`` equal slices of the flat array,
    slice i from the i-th PCG64 stream spawned from ``seed`` (filled in parallel
    threads; the values do not depend on the thread count)."""
    import concurrent.futures as cf
    import os
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    streams = np.random.SeedSequence(seed).spawn(chunks)
    bounds = [(i * n // chunks, (i + 1) * n // chunks) for i in range(chunks)]

    def fill(i):
        lo, hi = bounds[i]
        g = np.random.Generator(np.random.PCG64(streams[i]))
        draws = g.standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi] = to_f16_bits(draws) if dtype == F16 else to_bf16_bits(draws)

    with cf.ThreadPoolExecutor(max_workers=max(1, min(chunks, os.cpu_count() or 1))) as ex:
        list(ex.map(fill, range(chunks)))
    return out.reshape(shape)


def make_attention_case(seed: int, nq: int, n_kv_heads: int, capacity_tokens: int, tokens, k: int, *,
                        group: int = 16, ids: np.ndarray | None = None, n_valid=None,
                        name: str = "", dtype: int = BF16) -> AttnCase:
    """qa, kc, vc ~ N(0,1) (bf16, or fp16 with dtype F16), contexts ``tokens`` (scalar
    or per query); the ids are random distinct blocks of each context unless given."""
    rng = np.random.default_rng(seed)
    H = n_kv_heads * group
    draws = rng.standard_normal((nq, H, HEAD_DIM), dtype=np.float32)
    qa = to_f16_bits(draws) if dtype == F16 else to_bf16_bits(draws)
    kc = normal_16bit(seed + 2, (n_kv_heads, capacity_tokens, HEAD_DIM), dtype=dtype)
    vc = normal_16bit(seed + 3, (n_kv_heads, capacity_tokens, HEAD_DIM), dtype=dtype)
    toks = np.broadcast_to(np.asarray(tokens, dtype=np.int64), (nq,)).astype(np.int32)
    if ids is None:
        ids = random_ids(seed + 1, blocks_for_tokens(toks), k, n_valid)
    return AttnCase(qa=qa, kc=kc, vc=vc, ids=np.ascontiguousarray(ids, dtype=np.int32), n_tokens=toks,
                    scale=HEAD_DIM ** -0.5, name=name, dtype=dtype)


ATTN_KV_HEADS = 4


def deep_attention_case(ids: np.ndarray | None = None) -> AttnCase:
    """Selection attention at the deep prompt's depth: 256 queries x 64 heads (4 GQA
    groups of 16), bf16, capacity 524,288 tokens, contexts of 520,000 tokens, k = 32
    (random distinct blocks of the context unless ``ids`` are given)."""
    return make_attention_case(4100, 256, ATTN_KV_HEADS, 524_288, 520_000, 32, ids=ids,
                               name="deep prompt attention: 256q x 64 heads (4 groups of 16) bf16, "
                                    "520,000 tokens, capacity 524,288, k = 32")


def decode_attention_case(ids: np.ndarray | None = None) -> AttnCase:
    """Selection attention for a decode window: 3 queries x 64 heads (4 GQA groups of
    16), bf16, capacity 262,144 tokens, contexts of 258,000 tokens, k = 32."""
    return make_attention_case(2100, 3, ATTN_KV_HEADS, 262_144, 258_000, 32, ids=ids,
                               name="decode attention: 3q x 64 heads (4 groups of 16) bf16, "
                                    "258,000 tokens, capacity 262,144, k = 32")


def vcache_blocks_transposed(vc: np.ndarray) -> np.ndarray:
    """[Hkv, C, D] token rows -> [Hkv, C/64, D, 64]: each 64-token block of V stored
    dimension-major (the layout the CUDA selection attention reads)."""
    Hkv, C, D = vc.shape
    return np.ascontiguousarray(vc.reshape(Hkv, C // BLOCK_TOKENS, BLOCK_TOKENS, D).transpose(0, 1, 3, 2))
