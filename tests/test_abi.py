"""The C-ABI library (CPU side): it loads, exports every symbol include/qsa.h
declares, sizes workspaces, picks paths, and rejects bad arguments on the host
before any launch.  No kernel runs here."""
import ctypes
import os
import re

import pytest

from sparse_attention_kv_gb300 import _build, qsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qsa.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return qsa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert sorted(qsa.EXPORTS) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version(lib):
    assert lib.qsa_version() == 1


def test_workspace_sizes(lib):
    a = lib.qsa_workspace_bytes(256, 8192, 32, 0)
    assert a > 256 and a % 256 == 0
    assert lib.qsa_workspace_bytes(3, 4096, 32, 0) < a
    for bad in ((0, 8192, 32), (1, 0, 32), (1, 8192, 0), (1, 8192, 1025), (1, (1 << 24) + 1, 8)):
        assert lib.qsa_workspace_bytes(*bad, 0) == 0


def test_auto_path_rules(lib):
    # k <= 32 and rows of up to 8,192 blocks: the warp path, decode and prompt alike
    for nq, mb, act in ((3, 4096, -1), (16, 4096, -1), (256, 8192, 8125), (256, 2048, 2048), (256, 8192, 1000),
                        (1, 8192, -1)):
        assert lib.qsa_auto_path(nq, mb, act, 32) == qsa.PATH_WARP
        assert lib.qsa_auto_path(nq, mb, act, 1) == qsa.PATH_WARP
    # larger k: decode windows (no active count, few queries) split
    assert lib.qsa_auto_path(3, 4096, -1, 64) == qsa.PATH_SPLIT
    assert lib.qsa_auto_path(16, 4096, -1, 64) == qsa.PATH_SPLIT
    # prompt calls: sampled filter past the threshold, register below it
    assert lib.qsa_auto_path(256, 8192, 8125, 64) == qsa.PATH_SAMPLE
    assert lib.qsa_auto_path(256, 2048, 2048, 64) == qsa.PATH_SAMPLE
    assert lib.qsa_auto_path(256, 8192, 1000, 64) == qsa.PATH_REGISTER
    # beyond the on-chip reach: radix
    assert lib.qsa_auto_path(256, 100000, 100000, 32) == qsa.PATH_RADIX
    assert lib.qsa_auto_path(64, 100000, -1, 32) == qsa.PATH_RADIX
    assert lib.qsa_auto_path(256, 8193, 8193, 32) == qsa.PATH_RADIX


FAKE = 0x10000   # never dereferenced: each call below fails validation first


@pytest.mark.parametrize("case,status", [
    (dict(q=None), qsa.ERR_INVALID_ARG),
    (dict(head_dim=64), qsa.ERR_INVALID_ARG),
    (dict(n_heads=3), qsa.ERR_INVALID_ARG),
    (dict(n_heads=32), qsa.ERR_INVALID_ARG),
    (dict(nq=0), qsa.ERR_INVALID_ARG),
    (dict(max_blocks=0), qsa.ERR_INVALID_ARG),
    (dict(stride=100), qsa.ERR_INVALID_ARG),
    (dict(dt=7), qsa.ERR_INVALID_ARG),
    (dict(q=FAKE + 4), qsa.ERR_INVALID_ARG),
    (dict(active=-2), qsa.ERR_INVALID_ARG),
    (dict(k=0), qsa.ERR_INVALID_ARG),
    (dict(k=1025), qsa.ERR_INVALID_ARG),
    (dict(ws=None), qsa.ERR_WORKSPACE),
    (dict(ws_bytes=1024), qsa.ERR_WORKSPACE),
    (dict(ws=FAKE + 64), qsa.ERR_WORKSPACE),
])
def test_select_rejects_bad_arguments_before_launch(lib, case, status):
    a = dict(q=FAKE, w=FAKE, kblk=FAKE, dt=qsa.BF16, n_blocks=FAKE, nq=4, n_heads=16, head_dim=128,
             max_blocks=1024, active=-1, k=32, ids=FAKE, scores=FAKE, stride=1024, fused=0, ws=FAKE,
             ws_bytes=1 << 30, path=qsa.PATH_AUTO)
    a.update(case)
    st = lib.qsa_select(a["q"], a["w"], a["kblk"], a["dt"], a["n_blocks"], a["nq"], a["n_heads"],
                        a["head_dim"], a["max_blocks"], a["active"], a["k"], a["ids"], a["scores"],
                        a["stride"], a["fused"], a["ws"], a["ws_bytes"], a["path"], None)
    assert st == status
    assert lib.qsa_last_error().decode()


@pytest.mark.parametrize("case,status", [
    (dict(qa=None), qsa.ERR_INVALID_ARG),
    (dict(out=None), qsa.ERR_INVALID_ARG),
    (dict(nq=0), qsa.ERR_INVALID_ARG),
    (dict(head_dim=64), qsa.ERR_INVALID_ARG),
    (dict(n_heads=32), qsa.ERR_INVALID_ARG),      # not 16 x n_kv_heads
    (dict(n_kv=0, n_heads=0), qsa.ERR_INVALID_ARG),
    (dict(k=0), qsa.ERR_INVALID_ARG),
    (dict(k=65), qsa.ERR_INVALID_ARG),
    (dict(capacity=100), qsa.ERR_INVALID_ARG),
    (dict(capacity=0), qsa.ERR_INVALID_ARG),
    (dict(capacity=1 << 29, n_kv=2, n_heads=32), qsa.ERR_INVALID_ARG),
    (dict(kcache=FAKE + 8), qsa.ERR_INVALID_ARG),
    (dict(scale=0.0), qsa.ERR_INVALID_ARG),
    (dict(scale=float("inf")), qsa.ERR_INVALID_ARG),
    (dict(scale=float("nan")), qsa.ERR_INVALID_ARG),
    (dict(ws_bytes=16), qsa.ERR_WORKSPACE),
    (dict(ws=FAKE + 64), qsa.ERR_WORKSPACE),
    (dict(dt=qsa.F32), qsa.ERR_UNSUPPORTED),
    (dict(dt=qsa.E4M3), qsa.ERR_UNSUPPORTED),
    (dict(dt=9), qsa.ERR_UNSUPPORTED),
])
def test_select_attention_rejects_bad_arguments_before_launch(lib, case, status):
    a = dict(qa=FAKE, kcache=FAKE, vcache=FAKE, dt=qsa.BF16, ids=FAKE, k=32, n_tokens=FAKE, nq=4, n_heads=64,
             n_kv=4, head_dim=128, capacity=4096, scale=128 ** -0.5, out=FAKE, lse=FAKE, ws=FAKE, ws_bytes=256)
    a.update(case)
    st = lib.qsa_select_attention(a["qa"], a["kcache"], a["vcache"], a["dt"], a["ids"], a["k"], a["n_tokens"],
                                  a["nq"], a["n_heads"], a["n_kv"], a["head_dim"], a["capacity"], a["scale"],
                                  a["out"], a["lse"], a["ws"], a["ws_bytes"], None)
    assert st == status
    assert lib.qsa_last_error().decode()


@pytest.mark.parametrize("case", [
    dict(v=None), dict(v=FAKE + 2), dict(n_kv=0), dict(capacity=100), dict(capacity=0),
    dict(first=-1), dict(n=-1), dict(first=60, n=5), dict(vt=FAKE + 4096),   # overlapping buffers
    dict(n_kv=70000, capacity=64, n=1),   # more KV heads than a grid dimension holds
])
def test_vcache_transpose_rejects_bad_arguments(lib, case):
    a = dict(v=FAKE, vt=FAKE + (1 << 24), n_kv=2, capacity=4096, first=0, n=64)
    a.update(case)
    st = lib.qsa_vcache_transpose(a["v"], a["vt"], a["n_kv"], a["capacity"], a["first"], a["n"], None)
    assert st == qsa.ERR_INVALID_ARG
    assert lib.qsa_last_error().decode()


def test_topk_rejects_bad_arguments_before_launch(lib):
    st = lib.qsa_block_topk(FAKE, 100, FAKE, 4, 1024, -1, 32, FAKE, FAKE, 1 << 30, 0, None)
    assert st == qsa.ERR_INVALID_ARG   # stride < max_blocks
    st = lib.qsa_block_topk(FAKE, 1024, FAKE, 4, 1024, -1, 32, FAKE, FAKE, 16, 0, None)
    assert st == qsa.ERR_WORKSPACE
    st = lib.qsa_block_topk(None, 1024, FAKE, 4, 1024, -1, 32, FAKE, FAKE, 1 << 30, 0, None)
    assert st == qsa.ERR_INVALID_ARG
    st = lib.qsa_block_topk(FAKE, 1024, FAKE, 4, 1024, -1, 32, FAKE, FAKE, 1 << 30, 9, None)
    assert st == qsa.ERR_INVALID_ARG   # bad path enum


@pytest.mark.parametrize("case,status", [
    (dict(scores=None), qsa.ERR_INVALID_ARG),
    (dict(cand_scores=None), qsa.ERR_INVALID_ARG),
    (dict(cand_ids=None), qsa.ERR_INVALID_ARG),
    (dict(offset=-1), qsa.ERR_INVALID_ARG),
    (dict(offset=(1 << 31) - 1000), qsa.ERR_INVALID_ARG),   # ids past 2^31 - 1
    (dict(k=0), qsa.ERR_INVALID_ARG),
    (dict(k=1025), qsa.ERR_INVALID_ARG),
    (dict(nq=0), qsa.ERR_INVALID_ARG),
    (dict(stride=100), qsa.ERR_INVALID_ARG),
    (dict(active=-2), qsa.ERR_INVALID_ARG),
    (dict(ws_bytes=16), qsa.ERR_WORKSPACE),
    (dict(ws=None), qsa.ERR_WORKSPACE),
    (dict(path=9), qsa.ERR_INVALID_ARG),
])
def test_block_candidates_rejects_bad_arguments_before_launch(lib, case, status):
    a = dict(scores=FAKE, stride=1024, n_blocks=FAKE, nq=4, max_blocks=1024, active=-1, k=32, offset=4096,
             cand_scores=FAKE, cand_ids=FAKE, ws=FAKE, ws_bytes=1 << 30, path=qsa.PATH_AUTO)
    a.update(case)
    st = lib.qsa_block_candidates(a["scores"], a["stride"], a["n_blocks"], a["nq"], a["max_blocks"], a["active"],
                                  a["k"], a["offset"], a["cand_scores"], a["cand_ids"], a["ws"], a["ws_bytes"],
                                  a["path"], None)
    assert st == status
    assert lib.qsa_last_error().decode()


@pytest.mark.parametrize("case,status", [
    (dict(cs=None), qsa.ERR_INVALID_ARG),
    (dict(ci=None), qsa.ERR_INVALID_ARG),
    (dict(ids=None), qsa.ERR_INVALID_ARG),
    (dict(nq=0), qsa.ERR_INVALID_ARG),
    (dict(k=0), qsa.ERR_INVALID_ARG),
    (dict(k=1025), qsa.ERR_INVALID_ARG),
    (dict(g=0), qsa.ERR_INVALID_ARG),
    (dict(g=129, k=32), qsa.ERR_UNSUPPORTED),   # 4,128 candidates per query
    (dict(g=5, k=1024), qsa.ERR_UNSUPPORTED),
])
def test_merge_candidates_rejects_bad_arguments_before_launch(lib, case, status):
    a = dict(cs=FAKE, ci=FAKE, g=4, nq=8, k=32, ids=FAKE)
    a.update(case)
    st = lib.qsa_merge_candidates(a["cs"], a["ci"], a["g"], a["nq"], a["k"], a["ids"], None)
    assert st == status
    assert lib.qsa_last_error().decode()


def test_merge_capacity_matches_binding(lib):
    assert lib.qsa_merge_candidates(FAKE, FAKE, qsa.MERGE_CAP // 32 + 1, 1, 32, FAKE, None) == qsa.ERR_UNSUPPORTED


@pytest.mark.parametrize("args,status", [
    ((None, 1024, FAKE, 4, 1024, -1, 32, FAKE, 0), qsa.ERR_INVALID_ARG),
    ((FAKE, 100, FAKE, 4, 1024, -1, 32, FAKE, 0), qsa.ERR_INVALID_ARG),      # stride < max_blocks
    ((FAKE, 1024, FAKE, 4, 1024, -2, 32, FAKE, 0), qsa.ERR_INVALID_ARG),
    ((FAKE, 1024, FAKE, 4, 1024, -1, 32, FAKE, 9), qsa.ERR_INVALID_ARG),     # bad path
    ((FAKE, 1024, None, 4, 1024, -1, 32, FAKE, 0), qsa.ERR_INVALID_ARG),
    ((FAKE, 8192, FAKE, 256, 8192, -1, 1024, FAKE, 0), qsa.ERR_WORKSPACE),  # beyond the static scratch
])
def test_static_topk_rejects_before_touching_its_scratch(lib, args, status):
    """Rejected calls return before the scratch is looked up or cleared (no CUDA call
    at all, so this runs without a GPU)."""
    assert lib.qsa_block_topk_static(*args, None) == status
    assert lib.qsa_last_error().decode()


def test_binding_raises_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(qsa, "_lib", None)
    monkeypatch.setattr(qsa, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        qsa.load()
