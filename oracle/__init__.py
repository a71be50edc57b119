"""CPU oracle for query-sparse-attention block selection.

TEST INFRASTRUCTURE ONLY.  The parity tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` use it; the CUDA library never does.  It
shares no code with the GPU path: its arithmetic lives in ``qsa_oracle.c``
(plain C, IEEE double, full sort), compiled here with gcc and called through
ctypes.  This module only marshals numpy arrays.

Functions
---------
block_scores(q, w, kblk, n_blocks, dtype)
    Double-precision block scores, ``[nq, max_blocks]`` (entries at
    ``b >= n_blocks[q]`` are 0).  ``q``/``kblk`` are float32 arrays, or the bit
    patterns of bf16 or fp16 (uint16; fp16 by ``dtype`` only) or fp8 e4m3 (uint8).
select(scores, n_blocks, k)
    Per-query top-k over double scores: ids ascending, ties to the lower
    block id, -1 padded.
select_f32(scores, n_blocks, k)
    The same selection over float32 scores (e.g. the GPU's own).
select_attention(qa, kc, vc, ids, n_tokens, scale, dtype)
    Selection attention over the selected blocks in double: per query and
    head, softmax(scale * q.K^T) V over the tokens of the query's distinct
    selected blocks below its context length, and the log-sum-exp.  ``qa``
    [nq,H,D], ``kc``/``vc`` [Hkv,C,D] (token rows) as bf16 bits (uint16).

The parity rules (a)-(d) that compare the CUDA path's outputs with this
oracle's are in ``oracle.parity``.

Parity status: pinned (see the oracle tests).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB = os.path.join(_HERE, "libqsa_oracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1
E4M3 = 2
F16 = 3
_STORAGE = {F32: np.float32, BF16: np.uint16, E4M3: np.uint8, F16: np.uint16}


def build(force: bool = False) -> str:
    """Compile qsa_oracle.c into libqsa_oracle.so (gcc, -O2, no fast-math)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                   "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i32p = ctypes.POINTER(ctypes.c_int32)
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        vp = ctypes.c_void_p
        lib.qsa_oracle_block_scores.argtypes = [vp, fp, vp, ctypes.c_int, i32p, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int, dp]
        lib.qsa_oracle_block_scores.restype = ctypes.c_int
        lib.qsa_oracle_select.argtypes = [dp, ctypes.c_int64, i32p, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, i32p]
        lib.qsa_oracle_select.restype = ctypes.c_int
        lib.qsa_oracle_select_f32.argtypes = [fp, ctypes.c_int64, i32p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, i32p]
        lib.qsa_oracle_select_f32.restype = ctypes.c_int
        lib.qsa_oracle_select_attention.argtypes = [vp, vp, vp, ctypes.c_int, i32p, ctypes.c_int, i32p, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_double, dp, dp]
        lib.qsa_oracle_select_attention.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def block_scores(q: np.ndarray, w: np.ndarray, kblk: np.ndarray, n_blocks: np.ndarray,
                 dtype: int | None = None) -> np.ndarray:
    """Scores in double; q [nq,H,D], w [nq,H] fp32, kblk [C,D]; fp32, or bf16 (uint16) / e4m3 (uint8) bits."""
    lib = _load()
    if dtype is None:
        dtype = {np.dtype(np.uint16): BF16, np.dtype(np.uint8): E4M3}.get(np.asarray(q).dtype, F32)
    want = _STORAGE[dtype]
    q = np.ascontiguousarray(q, dtype=want)
    kblk = np.ascontiguousarray(kblk, dtype=want)
    w = np.ascontiguousarray(w, dtype=np.float32)
    n_blocks = np.ascontiguousarray(n_blocks, dtype=np.int32)
    nq, H, D = q.shape
    C = kblk.shape[0]
    if kblk.shape[1] != D or w.shape != (nq, H) or n_blocks.shape != (nq,):
        raise ValueError("oracle.block_scores: shape mismatch")
    out = np.zeros((nq, C), dtype=np.float64)
    rc = lib.qsa_oracle_block_scores(q.ctypes.data, _ptr(w, ctypes.c_float), kblk.ctypes.data,
                                     int(dtype), _ptr(n_blocks, ctypes.c_int32), nq, H, D, C,
                                     _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle.block_scores: bad argument")
    return out


def select(scores: np.ndarray, n_blocks: np.ndarray, k: int) -> np.ndarray:
    """Top-k ids [nq, k] over double scores [nq, C]."""
    lib = _load()
    scores = np.ascontiguousarray(scores, dtype=np.float64)
    n_blocks = np.ascontiguousarray(n_blocks, dtype=np.int32)
    nq, C = scores.shape
    ids = np.empty((nq, k), dtype=np.int32)
    rc = lib.qsa_oracle_select(_ptr(scores, ctypes.c_double), C, _ptr(n_blocks, ctypes.c_int32),
                               nq, C, int(k), _ptr(ids, ctypes.c_int32))
    if rc != 0:
        raise ValueError("oracle.select: bad argument")
    return ids


def select_f32(scores: np.ndarray, n_blocks: np.ndarray, k: int) -> np.ndarray:
    """Top-k ids [nq, k] over float32 scores [nq, C] (each widened exactly)."""
    lib = _load()
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    n_blocks = np.ascontiguousarray(n_blocks, dtype=np.int32)
    nq, C = scores.shape
    ids = np.empty((nq, k), dtype=np.int32)
    rc = lib.qsa_oracle_select_f32(_ptr(scores, ctypes.c_float), C,
                                   _ptr(n_blocks, ctypes.c_int32), nq, C, int(k),
                                   _ptr(ids, ctypes.c_int32))
    if rc != 0:
        raise ValueError("oracle.select_f32: bad argument")
    return ids


def select_attention(qa: np.ndarray, kc: np.ndarray, vc: np.ndarray, ids: np.ndarray,
                     n_tokens: np.ndarray, scale: float, dtype: int = BF16) -> tuple[np.ndarray, np.ndarray]:
    """(out [nq,H,D], lse [nq,H]) in double; qa [nq,H,D], kc/vc [Hkv,C,D] as bf16 or fp16
    bits (uint16, ``dtype``), ids [nq,k] int32."""
    lib = _load()
    qa = np.ascontiguousarray(qa, dtype=np.uint16)
    kc = np.ascontiguousarray(kc, dtype=np.uint16)
    vc = np.ascontiguousarray(vc, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n_tokens = np.ascontiguousarray(n_tokens, dtype=np.int32)
    nq, H, D = qa.shape
    Hkv, C, Dk = kc.shape
    k = ids.shape[1]
    if vc.shape != kc.shape or Dk != D or ids.shape[0] != nq or n_tokens.shape != (nq,):
        raise ValueError("oracle.select_attention: shape mismatch")
    out = np.zeros((nq, H, D), dtype=np.float64)
    lse = np.zeros((nq, H), dtype=np.float64)
    if dtype not in (BF16, F16):
        raise ValueError("oracle.select_attention: bf16 or fp16 inputs")
    rc = lib.qsa_oracle_select_attention(qa.ctypes.data, kc.ctypes.data, vc.ctypes.data, int(dtype),
                                         _ptr(ids, ctypes.c_int32), int(k), _ptr(n_tokens, ctypes.c_int32),
                                         nq, H, Hkv, D, C, float(scale), _ptr(out, ctypes.c_double),
                                         _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle.select_attention: bad argument")
    return out, lse
