"""Top-16 candidates of rows whose vocabulary is split over the ranks of a
process group (an LM head sharded by vocabulary): each rank reduces its slice
to a partial on its GPU, one all-gather exchanges the partials, and every rank
merges them into the whole rows' candidates, U and lse.

The pages run the drafter on one GPU (FreeToken PR 857, "Known gaps":
speculative decoding still needs --tp 1); this is an addition of the library
for a vocabulary-parallel LM head.  Argument marshalling and the exchange
only: the partial and the merge run in libdflash2.so.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding


def slice_bounds(V_total: int, world: int, rank: int) -> tuple[int, int]:
    """Token range [lo, hi) of `rank` when V_total tokens are split into `world` near-equal slices."""
    return rank * V_total // world, (rank + 1) * V_total // world


def sharded_topk16(logits_slice: torch.Tensor, id_offset: int, V_total: int, params=None, rows_per_param: int = 1,
                   group=None, shard_fn=None, merge_fn=None):
    """Candidates of the whole rows from this rank's slice of their logits.

    logits_slice [rows, Vs] holds tokens id_offset .. id_offset + Vs - 1 of every row; the ranks'
    slices must tile 0 .. V_total - 1.  Every rank gets the same (cand_idx, cand_U, lse).
    shard_fn / merge_fn default to the library's dflash2_topk16_shard / dflash2_topk16_merge; a
    test may pass others with the same signatures to exercise the exchange without a GPU.
    """
    shard_fn = shard_fn or binding.topk16_shard
    merge_fn = merge_fn or binding.topk16_merge
    part = shard_fn(logits_slice, id_offset, V_total, params=params, rows_per_param=rows_per_param)
    world = dist.get_world_size(group)
    stacked = []
    for t in part:
        t = t.contiguous()
        out = torch.empty((world * t.shape[0],) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        dist.all_gather_into_tensor(out, t, group=group)   # rank r's part at rows r * n .. (r + 1) * n
        stacked.append(out.view((world,) + tuple(t.shape)))
    return merge_fn(*stacked, V_total, params=params, rows_per_param=rows_per_param)
