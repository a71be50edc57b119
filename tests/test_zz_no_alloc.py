"""The allocation-free top-k entry point (qsa_block_topk_static).

Callers that may not allocate device memory where they select blocks -- a fixed
arena that must not grow, a plug-in given only its input and output buffers --
use qsa_block_topk_static, which takes its scratch from an array compiled into
the library.  Its ids must equal those of qsa_block_topk (the caller-workspace
entry point) bit for bit, and the oracle's selection over the same scores, on
consecutive calls that reuse the shared scratch.
This file is collected last, so a run that stops at its first failure has run
every other test before it.
"""
import ctypes

import numpy as np
import pytest

import oracle
from workloads import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from sparse_attention_kv_gb300 import qsa  # noqa: E402


def _call_static(lib, scores, n_dev, k, ids, max_blocks, active, path):
    return lib.qsa_block_topk_static(ctypes.c_void_p(scores.data_ptr()), scores.stride(0),
                                     ctypes.c_void_p(n_dev.data_ptr()), scores.shape[0], max_blocks, active, k,
                                     ctypes.c_void_p(ids.data_ptr()), path,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape", [
    (3, 4096, [4032, 626, 4096], 32, -1, qsa.PATH_AUTO),        # decode window: the warp path
    (3, 4096, [4032, 4000, 31], 32, -1, qsa.PATH_SPLIT),
    (128, 2048, None, 32, 2048, qsa.PATH_SAMPLE),               # prompt rows: sampled filter
    (16, 8192, None, 64, 8192, qsa.PATH_RADIX),
])
def test_static_entry_matches_workspace_entry_on_two_calls(shape):
    nq, C, lens, k, active, path = shape
    lib = qsa.load()
    rng = np.random.default_rng(9100 + C + nq)
    nb = np.array(lens if lens else rng.integers(k // 2, C + 1, size=nq), dtype=np.int32)
    n_dev = torch.from_numpy(nb).cuda()
    for call in range(2):
        sc = inputs.normal_scores(9000 + 10 * C + call, nq, C)
        scores = torch.from_numpy(sc).cuda()
        want = torch.full((nq, k), -5, dtype=torch.int32, device="cuda")
        ws = qsa.alloc_workspace(nq, C, k)
        qsa.block_topk(scores, n_dev, k, want, ws, max_blocks=C, active_blocks=active, path=path)
        got = torch.full((nq, k), -7, dtype=torch.int32, device="cuda")
        st = _call_static(lib, scores, n_dev, k, got, C, active, path)
        assert st == qsa.OK, lib.qsa_last_error().decode()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got.cpu().numpy(), want.cpu().numpy())
        # and both are the oracle's selection over the same scores
        np.testing.assert_array_equal(got.cpu().numpy(), oracle.select_f32(sc, nb, k))


def test_static_entry_leaves_device_memory_unchanged():
    """After one call (which loads the kernels and looks up the scratch's address), more
    calls take no device memory: the free bytes the driver reports do not move."""
    lib = qsa.load()
    nq, C, k = 64, 4096, 32
    sc = inputs.normal_scores(9300, nq, C)
    scores = torch.from_numpy(sc).cuda()
    nb = np.full(nq, C, dtype=np.int32)
    n_dev = torch.from_numpy(nb).cuda()
    ids = torch.empty((nq, k), dtype=torch.int32, device="cuda")
    assert _call_static(lib, scores, n_dev, k, ids, C, -1, qsa.PATH_AUTO) == qsa.OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        assert _call_static(lib, scores, n_dev, k, ids, C, -1, qsa.PATH_AUTO) == qsa.OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    np.testing.assert_array_equal(ids.cpu().numpy(), oracle.select_f32(sc, nb, k))


def test_static_entry_rejects_sizes_beyond_its_scratch():
    lib = qsa.load()
    nq, C, k = 256, 8192, 1024
    assert qsa.workspace_bytes(nq, C, k) > 8 << 20
    scores = torch.zeros((nq, C), device="cuda")
    n_dev = torch.full((nq,), C, dtype=torch.int32, device="cuda")
    ids = torch.zeros((nq, k), dtype=torch.int32, device="cuda")
    st = _call_static(lib, scores, n_dev, k, ids, C, -1, qsa.PATH_AUTO)
    assert st == qsa.ERR_WORKSPACE
    assert "static scratch" in lib.qsa_last_error().decode()
