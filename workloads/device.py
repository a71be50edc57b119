"""Copies of the synthetic workloads' arrays to the GPU (torch tensors of the
formats the library takes).  Bits are copied as they are; no arithmetic."""
from __future__ import annotations

import numpy as np

from . import inputs


def to_device(case, device="cuda"):
    """(q, w, kblk, n_blocks) of a selection case on the device, q and kblk in the
    case's format (fp32, bf16 or fp8 e4m3)."""
    import torch
    if case.dtype == inputs.BF16:
        q = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16)
        kb = torch.from_numpy(case.kblk.view(np.int16)).view(torch.bfloat16)
    elif case.dtype == inputs.E4M3:
        q = torch.from_numpy(case.q).view(torch.float8_e4m3fn)
        kb = torch.from_numpy(case.kblk).view(torch.float8_e4m3fn)
    else:
        q = torch.from_numpy(case.q)
        kb = torch.from_numpy(case.kblk)
    return (q.to(device).contiguous(), torch.from_numpy(case.w).to(device).contiguous(),
            kb.to(device).contiguous(), torch.from_numpy(case.n_blocks).to(device).contiguous())


def attn_to_device(case, device="cuda"):
    """(qa, kcache, vcache_t, ids, n_tokens) of a selection-attention case on the device."""
    import torch
    tdt = torch.float16 if case.dtype == inputs.F16 else torch.bfloat16

    def b16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt).to(device)
    return (b16(case.qa), b16(case.kc), b16(inputs.vcache_blocks_transposed(case.vc)),
            torch.from_numpy(case.ids).to(device), torch.from_numpy(case.n_tokens).to(device))
