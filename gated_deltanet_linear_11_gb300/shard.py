"""Host-side sharding of a packed batch across ranks (one process per GPU).

Sequences are independent under the gated delta rule, so a packed batch shards by
sequence with no exchange on the data path: each rank runs its own sub-batch, and each
sequence's result is bit-identical to running it anywhere else (the kernels' math never
depends on the batch).  The only collective is the max-over-ranks of a timing.
"""
from __future__ import annotations

import numpy as np


def partition_sequences(lens, world):
    """Assign sequences to `world` ranks, balancing tokens (longest first, ties by index,
    each to the least-loaded rank, ties by rank).  Deterministic.  Returns a list of
    sorted sequence-index lists, one per rank."""
    lens = [int(x) for x in lens]
    order = sorted(range(len(lens)), key=lambda i: (-lens[i], i))
    load = [0] * world
    parts = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda k: (load[k], k))
        parts[r].append(i)
        load[r] += lens[i]
    return [sorted(p) for p in parts]


def sub_batch(cu_seqlens, seq_ids):
    """Token indices and offsets of the packed sub-batch made of `seq_ids` (in order).

    Returns (token_index int64 [T_sub], cu_sub int32 [len(seq_ids)+1])."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    idx = [np.arange(cu[i], cu[i + 1]) for i in seq_ids]
    tok = np.concatenate(idx) if idx else np.zeros(0, np.int64)
    cu_sub = np.zeros(len(seq_ids) + 1, np.int32)
    cu_sub[1:] = np.cumsum([cu[i + 1] - cu[i] for i in seq_ids])
    return tok, cu_sub


def max_over_ranks(value, device="cpu"):
    """MAX of a float over the default process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
