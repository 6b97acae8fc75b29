"""Vocabulary sharding of the local two-stage head over several GPUs.

The local Top-k of the EAGLE-4 notes ("A Local Top-k based variant") picks
each tile's candidates from that tile alone. Splitting the shuffled
positions into contiguous ranges of whole tiles therefore splits the work
with no exchange during selection: every GPU streams only its rows of A and
gathers only its own candidates' rows of W. The softmax over a row's
candidates is the one step that spans the shards, and it needs 8 bytes per
row from every shard: (max, sum of exponentials), exchanged by an all-gather
on the caller's process group (NCCL between GPUs). The kernels are
lmhead_shard_two_stage and lmhead_shard_softmax (include/lmhead.h).

    ranges = shard_ranges(n, T, world)
    W_s, A_s, tok_s, row_of_id = shard_inputs(W_bits, A_bits, token_ids, *ranges[rank])  # offline
    ids, logits, q = sharded_two_stage(W_s, A_s, B, h, tok_s, row_of_id, T, k_tile)      # per call
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import shard_softmax, shard_two_stage

__all__ = ["shard_ranges", "shard_inputs", "gather_stats", "sharded_two_stage"]


def shard_ranges(n: int, T: int, shards: int):
    """Contiguous position ranges [p0, p1), one per shard, each of whole tiles
    of T positions (the last one holds the head's short last tile); shards
    beyond the number of tiles get empty ranges."""
    if n < 1 or T < 1 or shards < 1:
        raise ValueError("n, T and shards must be positive")
    tiles = -(-n // T)
    per = -(-tiles // shards)
    return [(min(n, g * per * T), min(n, (g + 1) * per * T)) for g in range(shards)]


def shard_inputs(W_bits: np.ndarray, A_bits: np.ndarray, token_ids: np.ndarray, p0: int, p1: int):
    """Offline: one shard's inputs from the whole head (host arrays; A in the
    shuffled position order, token_ids position -> vocabulary id). Returns
    (W_shard, A_shard, token_ids_shard, row_of_id)."""
    n = W_bits.shape[0]
    tok = np.ascontiguousarray(token_ids[p0:p1], dtype=np.int32)
    row_of_id = np.full(n, -1, dtype=np.int32)
    row_of_id[tok] = np.arange(p1 - p0, dtype=np.int32)
    return (np.ascontiguousarray(W_bits[tok]), np.ascontiguousarray(A_bits[p0:p1]), tok,
            row_of_id)


def gather_stats(stats: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather every shard's M x 2 stats over the process group, in rank
    order: G x M x 2 (without an initialised process group: this shard's
    alone)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return stats.unsqueeze(0)
    world = dist.get_world_size(group)
    parts = [torch.empty_like(stats) for _ in range(world)]
    dist.all_gather(parts, stats.contiguous(), group=group)
    return torch.stack(parts)


def sharded_two_stage(W_shard, A_shard, B, h, token_ids_shard, row_of_id, T: int, k_tile: int,
                      temperature: float = 1.0, group=None, workspace=None,
                      stream: Optional[torch.cuda.Stream] = None):
    """This rank's shard of the local head: its candidates' vocabulary ids,
    exact logits and their q under the softmax over every shard's candidates.
    Concatenating the ranks' outputs (rank order) gives the unsharded head's
    candidates in tile order when every shard holds whole tiles."""
    ids, logits, stats = shard_two_stage(W_shard, A_shard, B, h, token_ids_shard, row_of_id, T,
                                         k_tile, temperature, workspace=workspace, stream=stream)
    all_stats = gather_stats(stats, group)
    q = shard_softmax(all_stats, logits, temperature, stream=stream)
    return ids, logits, q
