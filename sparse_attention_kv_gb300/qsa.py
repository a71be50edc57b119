"""ctypes binding of libqsa.so (include/qsa.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module checks
tensor placement, passes raw device pointers, sizes and the current CUDA
stream, and turns error statuses into exceptions.  PyTorch supplies device
memory and streams.  There is no fallback: if libqsa.so is missing or fails
to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqsa.so")

# qsa_status
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = range(5)
# qsa_dtype
F32, BF16, E4M3, F16 = 0, 1, 2, 3
# qsa_path
PATH_AUTO, PATH_SPLIT, PATH_SAMPLE, PATH_REGISTER, PATH_RADIX, PATH_WARP = range(6)
PATH_NAMES = {PATH_AUTO: "auto", PATH_SPLIT: "split", PATH_SAMPLE: "sample",
              PATH_REGISTER: "register", PATH_RADIX: "radix", PATH_WARP: "warp"}
# flags word bits
FLAG_NBLOCKS_CLAMPED, FLAG_WAIT_TIMEOUT, FLAG_INTERNAL, FLAG_SAMPLE_FALLBACK = 0x1, 0x2, 0x4, 0x8
FLAG_BAD_ID = 0x10
ERROR_FLAGS = FLAG_NBLOCKS_CLAMPED | FLAG_WAIT_TIMEOUT | FLAG_INTERNAL | FLAG_BAD_ID
HEAD_DIM = 128
MAX_K = 1024
ATTN_GROUP = 16
ATTN_MAX_K = 64

EXPORTS = ("qsa_workspace_bytes", "qsa_workspace_init", "qsa_block_scores", "qsa_block_topk",
           "qsa_block_topk_static", "qsa_block_candidates", "qsa_merge_candidates", "qsa_select",
           "qsa_select_attention", "qsa_vcache_transpose", "qsa_read_flags", "qsa_auto_path", "qsa_last_error",
           "qsa_version")
MERGE_CAP = 4096   # candidates per query qsa_merge_candidates holds (n_shards x k)


class QSAError(RuntimeError):
    def __init__(self, fn: str, status: int, reason: str):
        super().__init__(f"{fn} failed with status {status}: {reason}")
        self.status = status
        self.reason = reason


_lib = None


def load() -> ctypes.CDLL:
    """Load libqsa.so (built in-tree); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -m sparse_attention_kv_gb300._build` "
                           "(or __graft_entry__.build()) on a machine with nvcc")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.qsa_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.qsa_workspace_bytes.restype = sz
    lib.qsa_workspace_init.argtypes = [vp, sz, vp]
    lib.qsa_workspace_init.restype = i32
    lib.qsa_block_scores.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, vp, i64, vp, sz, vp]
    lib.qsa_block_scores.restype = i32
    lib.qsa_block_topk.argtypes = [vp, i64, vp, i32, i32, i32, i32, vp, vp, sz, i32, vp]
    lib.qsa_block_topk.restype = i32
    lib.qsa_block_topk_static.argtypes = [vp, i64, vp, i32, i32, i32, i32, vp, i32, vp]
    lib.qsa_block_topk_static.restype = i32
    lib.qsa_block_candidates.argtypes = [vp, i64, vp, i32, i32, i32, i32, i32, vp, vp, vp, sz, i32, vp]
    lib.qsa_block_candidates.restype = i32
    lib.qsa_merge_candidates.argtypes = [vp, vp, i32, i32, i32, vp, vp]
    lib.qsa_merge_candidates.restype = i32
    lib.qsa_select.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, vp, vp, i64, i32, vp,
                               sz, i32, vp]
    lib.qsa_select.restype = i32
    lib.qsa_select_attention.argtypes = [vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32, i32,
                                         ctypes.c_float, vp, vp, vp, sz, vp]
    lib.qsa_select_attention.restype = i32
    lib.qsa_vcache_transpose.argtypes = [vp, vp, i32, i32, i32, i32, vp]
    lib.qsa_vcache_transpose.restype = i32
    lib.qsa_read_flags.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), i32, vp]
    lib.qsa_read_flags.restype = i32
    lib.qsa_auto_path.argtypes = [i32, i32, i32, i32]
    lib.qsa_auto_path.restype = i32
    lib.qsa_last_error.argtypes = []
    lib.qsa_last_error.restype = ctypes.c_char_p
    lib.qsa_version.argtypes = []
    lib.qsa_version.restype = i32
    _lib = lib
    return lib


def _check(fn: str, status: int) -> None:
    if status != OK:
        raise QSAError(fn, status, load().qsa_last_error().decode(errors="replace"))


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dptr(t: torch.Tensor | None, name: str) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor, name: str) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    if t.dtype == getattr(torch, "float8_e4m3fn", None):
        return E4M3
    raise ValueError(f"{name} must be bfloat16, float32 or float8_e4m3fn (got {t.dtype})")


def _contig(t: torch.Tensor, name: str) -> None:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def version() -> int:
    return load().qsa_version()


def workspace_bytes(nq: int, max_blocks: int, k: int, fused: bool = False) -> int:
    return int(load().qsa_workspace_bytes(nq, max_blocks, k, int(bool(fused))))


def alloc_workspace(nq: int, max_blocks: int, k: int, device=None, fused: bool = False) -> torch.Tensor:
    """A zero-filled workspace (uint8 CUDA tensor) sized for these shapes."""
    n = workspace_bytes(nq, max_blocks, k, fused)
    if n == 0:
        raise ValueError("invalid workspace sizes")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def auto_path(nq: int, max_blocks: int, active_blocks: int, k: int) -> int:
    return int(load().qsa_auto_path(nq, max_blocks, active_blocks, k))


def block_scores(q: torch.Tensor, w: torch.Tensor, kblk: torch.Tensor, n_blocks: torch.Tensor,
                 scores: torch.Tensor, active_blocks: int = -1, ws: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """scores[q, b] for b < n_blocks[q]; q [nq,H,128], w [nq,H] fp32, kblk [C,128]
    (q and kblk both float32, bfloat16 or float8_e4m3fn)."""
    lib = load()
    for t, nm in ((q, "q"), (w, "w"), (kblk, "kblk"), (n_blocks, "n_blocks")):
        _contig(t, nm)
    nq, H, D = q.shape
    dt = _dtype_code(q, "q")
    if kblk.dtype != q.dtype or w.dtype != torch.float32 or n_blocks.dtype != torch.int32:
        raise ValueError("kblk must match q's dtype; w fp32; n_blocks int32")
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be a 2-D fp32 tensor with unit inner stride")
    st = lib.qsa_block_scores(_dptr(q, "q"), _dptr(w, "w"), _dptr(kblk, "kblk"), dt,
                              _dptr(n_blocks, "n_blocks"), nq, H, D, kblk.shape[0], active_blocks,
                              _dptr(scores, "scores"), scores.stride(0), _dptr(ws, "ws"),
                              0 if ws is None else ws.numel(), _stream(stream))
    _check("qsa_block_scores", st)
    return scores


def block_topk(scores: torch.Tensor, n_blocks: torch.Tensor, k: int, ids: torch.Tensor,
               ws: torch.Tensor, max_blocks: int | None = None, active_blocks: int = -1,
               path: int = PATH_AUTO, stream=None) -> torch.Tensor:
    """ids [nq, k] (int32, ascending, -1 padded) of the top-k blocks per query."""
    lib = load()
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be a 2-D fp32 tensor with unit inner stride")
    if ids.dtype != torch.int32 or not ids.is_contiguous() or tuple(ids.shape) != (scores.shape[0], k):
        raise ValueError("ids must be a contiguous int32 tensor [nq, k]")
    _contig(n_blocks, "n_blocks")
    nq = scores.shape[0]
    mb = scores.shape[1] if max_blocks is None else max_blocks
    st = lib.qsa_block_topk(_dptr(scores, "scores"), scores.stride(0), _dptr(n_blocks, "n_blocks"), nq,
                            mb, active_blocks, k, _dptr(ids, "ids"), _dptr(ws, "ws"), ws.numel(),
                            path, _stream(stream))
    _check("qsa_block_topk", st)
    return ids


def block_topk_static(scores: torch.Tensor, n_blocks: torch.Tensor, k: int, ids: torch.Tensor,
                      max_blocks: int | None = None, active_blocks: int = -1, path: int = PATH_AUTO,
                      stream=None) -> torch.Tensor:
    """block_topk without a workspace argument: the library's static scratch is used
    (for callers that may not allocate device memory)."""
    lib = load()
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be a 2-D fp32 tensor with unit inner stride")
    if ids.dtype != torch.int32 or not ids.is_contiguous() or tuple(ids.shape) != (scores.shape[0], k):
        raise ValueError("ids must be a contiguous int32 tensor [nq, k]")
    _contig(n_blocks, "n_blocks")
    nq = scores.shape[0]
    mb = scores.shape[1] if max_blocks is None else max_blocks
    st = lib.qsa_block_topk_static(_dptr(scores, "scores"), scores.stride(0), _dptr(n_blocks, "n_blocks"), nq,
                                   mb, active_blocks, k, _dptr(ids, "ids"), path, _stream(stream))
    _check("qsa_block_topk_static", st)
    return ids


def block_candidates(scores: torch.Tensor, n_blocks: torch.Tensor, k: int, cand_scores: torch.Tensor,
                     cand_ids: torch.Tensor, ws: torch.Tensor, block_offset: int, max_blocks: int | None = None,
                     active_blocks: int = -1, path: int = PATH_AUTO, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """One shard's candidates: cand_ids [nq, k] (global ids = block_offset + local id,
    ascending, -1 padded) and cand_scores [nq, k] fp32, over scores [nq, >= max_blocks]."""
    lib = load()
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be a 2-D fp32 tensor with unit inner stride")
    nq = scores.shape[0]
    if cand_ids.dtype != torch.int32 or not cand_ids.is_contiguous() or tuple(cand_ids.shape) != (nq, k):
        raise ValueError("cand_ids must be a contiguous int32 tensor [nq, k]")
    if cand_scores.dtype != torch.float32 or not cand_scores.is_contiguous() or tuple(cand_scores.shape) != (nq, k):
        raise ValueError("cand_scores must be a contiguous fp32 tensor [nq, k]")
    _contig(n_blocks, "n_blocks")
    mb = scores.shape[1] if max_blocks is None else max_blocks
    st = lib.qsa_block_candidates(_dptr(scores, "scores"), scores.stride(0), _dptr(n_blocks, "n_blocks"), nq, mb,
                                  active_blocks, k, int(block_offset), _dptr(cand_scores, "cand_scores"),
                                  _dptr(cand_ids, "cand_ids"), _dptr(ws, "ws"), ws.numel(), path, _stream(stream))
    _check("qsa_block_candidates", st)
    return cand_scores, cand_ids


def merge_candidates(cand_scores: torch.Tensor, cand_ids: torch.Tensor, ids: torch.Tensor,
                     stream=None) -> torch.Tensor:
    """ids [nq, k] (ascending, -1 padded) selected over every shard's candidates
    cand_scores / cand_ids [n_shards, nq, k]."""
    lib = load()
    if cand_scores.dim() != 3 or cand_scores.dtype != torch.float32 or not cand_scores.is_contiguous():
        raise ValueError("cand_scores must be a contiguous fp32 tensor [n_shards, nq, k]")
    if cand_ids.dtype != torch.int32 or not cand_ids.is_contiguous() or cand_ids.shape != cand_scores.shape:
        raise ValueError("cand_ids must be a contiguous int32 tensor shaped like cand_scores")
    G, nq, k = cand_scores.shape
    if ids.dtype != torch.int32 or not ids.is_contiguous() or tuple(ids.shape) != (nq, k):
        raise ValueError("ids must be a contiguous int32 tensor [nq, k]")
    st = lib.qsa_merge_candidates(_dptr(cand_scores, "cand_scores"), _dptr(cand_ids, "cand_ids"), G, nq, k,
                                  _dptr(ids, "ids"), _stream(stream))
    _check("qsa_merge_candidates", st)
    return ids


def select(q: torch.Tensor, w: torch.Tensor, kblk: torch.Tensor, n_blocks: torch.Tensor, k: int,
           ids: torch.Tensor, ws: torch.Tensor, scores: torch.Tensor | None = None,
           fused: bool = False, active_blocks: int = -1, path: int = PATH_AUTO,
           stream=None) -> torch.Tensor:
    """Score then select (chained: `scores` required; fused: optional debug copy)."""
    lib = load()
    for t, nm in ((q, "q"), (w, "w"), (kblk, "kblk"), (n_blocks, "n_blocks"), (ids, "ids")):
        _contig(t, nm)
    nq, H, D = q.shape
    dt = _dtype_code(q, "q")
    if scores is not None and (scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1):
        raise ValueError("scores must be a 2-D fp32 tensor with unit inner stride")
    st = lib.qsa_select(_dptr(q, "q"), _dptr(w, "w"), _dptr(kblk, "kblk"), dt, _dptr(n_blocks, "n_blocks"),
                        nq, H, D, kblk.shape[0], active_blocks, k, _dptr(ids, "ids"),
                        _dptr(scores, "scores"), 0 if scores is None else scores.stride(0),
                        int(bool(fused)), _dptr(ws, "ws"), ws.numel(), path, _stream(stream))
    _check("qsa_select", st)
    return ids


def select_attention(qa: torch.Tensor, kcache: torch.Tensor, vcache_t: torch.Tensor, ids: torch.Tensor,
                     n_tokens: torch.Tensor, out: torch.Tensor, lse: torch.Tensor | None = None,
                     scale: float | None = None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Selection attention over ids [nq, k]: out [nq, H, 128] fp32 (and lse [nq, H]).

    qa [nq, H, 128], kcache [Hkv, C, 128], vcache_t [Hkv, C/64, 128, 64] (each block of V
    dimension-major), all bfloat16 or all float16; n_tokens [nq] int32; H = 16 * Hkv."""
    lib = load()
    for t, nm in ((qa, "qa"), (kcache, "kcache"), (vcache_t, "vcache_t"), (ids, "ids"), (n_tokens, "n_tokens"),
                  (out, "out")):
        _contig(t, nm)
    if qa.dtype not in (torch.bfloat16, torch.float16) or kcache.dtype != qa.dtype or vcache_t.dtype != qa.dtype:
        raise ValueError("qa, kcache and vcache_t must all be bfloat16 or all float16")
    if ids.dtype != torch.int32 or n_tokens.dtype != torch.int32:
        raise ValueError("ids and n_tokens must be int32")
    nq, H, D = qa.shape
    Hkv, C, _ = kcache.shape
    if tuple(vcache_t.shape) != (Hkv, C // 64, D, 64):
        raise ValueError("vcache_t must be [n_kv_heads, capacity / 64, 128, 64]")
    if out.dtype != torch.float32 or tuple(out.shape) != (nq, H, D):
        raise ValueError("out must be a contiguous fp32 tensor [nq, n_heads, 128]")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (nq, H) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 tensor [nq, n_heads]")
    if scale is None:
        scale = D ** -0.5
    st = lib.qsa_select_attention(_dptr(qa, "qa"), _dptr(kcache, "kcache"), _dptr(vcache_t, "vcache_t"),
                                  F16 if qa.dtype == torch.float16 else BF16,
                                  _dptr(ids, "ids"), ids.shape[1], _dptr(n_tokens, "n_tokens"), nq, H, Hkv, D, C,
                                  float(scale), _dptr(out, "out"), _dptr(lse, "lse"), _dptr(ws, "ws"),
                                  0 if ws is None else ws.numel(), _stream(stream))
    _check("qsa_select_attention", st)
    return out


def vcache_transpose(v: torch.Tensor, vcache_t: torch.Tensor, first_block: int = 0, n_blocks: int | None = None,
                     stream=None) -> torch.Tensor:
    """vcache_t [Hkv, C/64, 128, 64] from v [Hkv, C, 128] (bf16 or fp16) for blocks
    [first_block, first_block + n_blocks) (all by default)."""
    lib = load()
    _contig(v, "v")
    _contig(vcache_t, "vcache_t")
    if v.dtype not in (torch.bfloat16, torch.float16) or vcache_t.dtype != v.dtype:
        raise ValueError("v and vcache_t must both be bfloat16 or both float16")
    Hkv, C, D = v.shape
    if D != 128 or tuple(vcache_t.shape) != (Hkv, C // 64, 128, 64):
        raise ValueError("v must be [Hkv, C, 128] and vcache_t [Hkv, C/64, 128, 64]")
    if n_blocks is None:
        n_blocks = C // 64 - first_block
    st = lib.qsa_vcache_transpose(_dptr(v, "v"), _dptr(vcache_t, "vcache_t"), Hkv, C, first_block, n_blocks,
                                  _stream(stream))
    _check("qsa_vcache_transpose", st)
    return vcache_t


def read_flags(ws: torch.Tensor, clear: bool = True, stream=None) -> int:
    """The workspace flags word (FLAG_* bits); waits for the stream."""
    out = ctypes.c_uint32(0)
    st = load().qsa_read_flags(_dptr(ws, "ws"), ctypes.byref(out), int(bool(clear)), _stream(stream))
    _check("qsa_read_flags", st)
    return int(out.value)
