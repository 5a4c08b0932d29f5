"""Indexer context parallelism over torch.distributed ranks.

"[MiniMax-M3.1] FP4 index cache and NVFP4 sparse KV cache" (ROCm/ATOM #2744),
review thread on the unused page-16 tables: with indexer CP one long request's
index keys are split over ranks, each rank scores its share, and the ranks'
candidate keys are merged (merge_candidate_keys) into the top-k. Here every
rank holds a contiguous slice of each request's blocks (its own pages and
block table); the scoring and the merge are the library's kernels, the
exchange is one all-gather of the ranks' [R, topk] candidate keys.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding as M


def exchange_candidates(local_keys: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's candidate keys, int64 [world, R, topk], from this rank's
    [R, topk] (an all-gather over ``group``; rank order)."""
    world = dist.get_world_size(group)
    local_keys = local_keys.contiguous()
    parts = [torch.empty_like(local_keys) for _ in range(world)]
    dist.all_gather(parts, local_keys, group=group)
    return torch.stack(parts)


def cp_index_score_topk(q_idx, w, codes, scales, block_table, blk_begin, blk_count, row_req, row_len,
                        topk: int, group=None, ws=None, err=None, init_blocks: int = 0,
                        local_blocks: int = 0):
    """The rows' top-k block ids over every rank's slice: this rank's candidates
    (m3s_index_score_candidates on its slice), all ranks' exchanged, merged
    (m3s_merge_candidates). Every rank returns the same ids."""
    local = M.m3s_index_score_candidates(q_idx, w, codes, scales, block_table, blk_begin, blk_count,
                                         row_req, row_len, topk, ws=ws, err=err,
                                         init_blocks=init_blocks, local_blocks=local_blocks)
    return M.m3s_merge_candidates(exchange_candidates(local, group), None)
