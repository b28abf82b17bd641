"""Vocabulary-sharded draft head with the local-argmax exchange ("q38_draft.py",
install: speculative_config.use_local_argmax_reduction; "FP8 MTP draft stack
...", ParallelLMHead, which splits the head's rows over ranks).

Each rank holds a contiguous range of the kept rows of one quantised head (the
global scale is the whole head's, so a shard's logits are the unsharded head's
logits of those rows). A draft step runs the rank's shard and produces one
int64 key per draft (draft_head_top_keys); one all-reduce(MAX) of M int64 over
the ranks picks the whole head's argmax (largest logit, then lowest id), which
draft_head_keys_to_ids turns into target ids. compute_logits writes each
shard's logits into a -inf row; an all-reduce(MAX) of the rows assembles the
full-vocabulary row (every id is written by one shard, -inf is the identity).

Host-side plumbing only: the step and the decode run in the library's kernels;
torch.distributed carries the 8-byte keys (NCCL on GPUs, gloo on CPUs).
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import DH_FMT_NVFP4, DH_FMT_NVFP4_PACKED, DraftHead, keys_to_ids, nvfp4_pack_head


class ShardExchangeError(RuntimeError):
    """The key exchange with the other ranks failed (a rank left, a timeout)."""


def shard_rows(n_kept: int, rank: int, world: int) -> tuple[int, int]:
    """Kept rows [lo, hi) of `rank`'s shard: contiguous, sizes within one."""
    if not (0 <= rank < world) or world > n_kept:
        raise ValueError(f"rank {rank} of {world} shards over {n_kept} kept rows")
    return rank * n_kept // world, (rank + 1) * n_kept // world


def shard_keep_mask(keep: np.ndarray, rank: int, world: int) -> np.ndarray:
    """The keep mask of `rank`'s shard: its range of the kept ids."""
    kept = np.flatnonzero(np.asarray(keep))
    lo, hi = shard_rows(kept.size, rank, world)
    out = np.zeros(np.asarray(keep).shape, dtype=np.uint8)
    out[kept[lo:hi]] = 1
    return out


def nvfp4_shard(q: torch.Tensor, sf: torch.Tensor, g: torch.Tensor, idx: torch.Tensor, n_kept: int, V: int,
                rank: int, world: int, packed: bool = True) -> DraftHead:
    """`rank`'s shard of an NVFP4 head quantised whole (q [N][K/2], sf [N][K/16],
    g, dh_idx ascending): its kept rows, padded to a multiple of 64 rows with
    copies of its first row (as the pages pad dh_idx), sharing g."""
    lo, hi = shard_rows(n_kept, rank, world)
    n = hi - lo
    rows = torch.arange(lo, hi, device=q.device)
    rows = torch.cat([rows, torch.full(((-n) % 64,), lo, dtype=rows.dtype, device=q.device)])
    q_s, sf_s, idx_s = q[rows].contiguous(), sf[rows].contiguous(), idx[rows].contiguous()
    if packed:
        return DraftHead(DH_FMT_NVFP4_PACKED, V, nvfp4_pack_head(q_s, sf_s), idx_s, n, scale=g, idx_ascending=True)
    return DraftHead(DH_FMT_NVFP4, V, q_s, idx_s, n, sf=sf_s, scale=g, idx_ascending=True)


def exchange_keys(keys: torch.Tensor, group=None) -> torch.Tensor:
    """In place: the maximum of every rank's keys (one all-reduce of M int64)."""
    try:
        dist.all_reduce(keys, op=dist.ReduceOp.MAX, group=group)
    except Exception as e:  # a rank that left or never joined, a timeout
        raise ShardExchangeError(f"argmax key exchange failed: {e}") from e
    return keys


class ShardedDraftHead:
    """This rank's shard plus the process group of all shards."""

    def __init__(self, shard: DraftHead, group=None):
        if shard.idx is not None and not shard.flags & 1:
            raise ValueError("a shard needs an ascending dh_idx (its keys carry target ids)")
        self.shard, self.group = shard, group

    def top_tokens(self, h: torch.Tensor, ids: torch.Tensor | None = None, top: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
        keys = self.shard.top_keys(h, stream=stream)
        exchange_keys(keys, self.group)
        return keys_to_ids(keys, ids, top, stream)

    def compute_logits(self, h: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        out = self.shard.compute_logits(h, out, stream)
        try:
            dist.all_reduce(out, op=dist.ReduceOp.MAX, group=self.group)
        except Exception as e:
            raise ShardExchangeError(f"logits exchange failed: {e}") from e
        return out
