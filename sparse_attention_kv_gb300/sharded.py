"""KV-sharded block selection across ranks (one GPU each).

Each rank holds a contiguous range of every query's KV blocks: their key rows,
and so their scores.  The selection is the same as one call over all blocks:

  1. stage A on each rank: qsa_block_candidates over the rank's score rows, with
     the range's first global block id as the offset -> [nq, k] candidates
     (score, global id);
  2. an all-gather of the candidates, nq * k * 8 bytes per rank, into the
     shard-major [world, nq, k] layout;
  3. stage B on every rank: qsa_merge_candidates -> ids [nq, k].

A query's selection restricted to one rank's blocks is a prefix of that range's
order (score descending, block id ascending), so the union of the ranks'
candidates holds every selected block (Strata PR #3987, section "Approach").
This module only moves tensors between the library's calls and the process
group; every selection step runs in libqsa.so.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import qsa


def _all_gather(t: torch.Tensor, world: int, group) -> torch.Tensor:
    out = torch.empty((world, *t.shape), dtype=t.dtype, device=t.device)
    if dist.get_backend(group) == "nccl":
        dist.all_gather_into_tensor(out, t, group=group)
    else:
        dist.all_gather(list(out.unbind(0)), t, group=group)
    return out


def select_kv_sharded(scores: torch.Tensor, n_blocks: torch.Tensor, k: int, block_offset: int, ids: torch.Tensor,
                      ws: torch.Tensor | None = None, max_blocks: int | None = None, active_blocks: int = -1,
                      group=None, stage_a=None, stage_b=None) -> torch.Tensor:
    """ids [nq, k] (ascending global block ids, -1 padded) selected over every rank's
    blocks.  scores [nq, >= max_blocks] are this rank's rows (local block ids), n_blocks
    [nq] int32 its per-query block counts, block_offset its first global block id.

    stage_a(scores, n_blocks, k, cand_scores, cand_ids, ws, block_offset, max_blocks,
    active_blocks) and stage_b(all_scores, all_ids, ids) default to the library's
    qsa.block_candidates and qsa.merge_candidates."""
    world = dist.get_world_size(group)
    nq = scores.shape[0]
    cand_scores = torch.empty((nq, k), dtype=torch.float32, device=scores.device)
    cand_ids = torch.empty((nq, k), dtype=torch.int32, device=scores.device)
    if stage_a is None:
        qsa.block_candidates(scores, n_blocks, k, cand_scores, cand_ids, ws, block_offset=block_offset,
                             max_blocks=max_blocks, active_blocks=active_blocks)
    else:
        stage_a(scores, n_blocks, k, cand_scores, cand_ids, ws, block_offset, max_blocks, active_blocks)
    all_scores = _all_gather(cand_scores, world, group)
    all_ids = _all_gather(cand_ids, world, group)
    if stage_b is None:
        qsa.merge_candidates(all_scores, all_ids, ids)
    else:
        stage_b(all_scores, all_ids, ids)
    return ids
