"""Data-parallel placement of GDN work across ranks (one GPU per rank).

The core has no exchange step: sequences (and value heads) are independent, so a
packed batch is split by whole sequences and each rank runs its share with no
collective on the data path.  Only timing uses a collective (max over ranks).
"""
from __future__ import annotations

import heapq

import numpy as np


def partition_sequences(lengths, world_size: int) -> list[list[int]]:
    """Assign sequence indices to ranks, balancing token counts.

    Longest-first greedy: each sequence goes to the rank with the fewest tokens
    so far (ties to the lower rank).  Deterministic; every sequence appears on
    exactly one rank; each rank's list is in ascending sequence order.
    """
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    lengths = [int(v) for v in lengths]
    order = sorted(range(len(lengths)), key=lambda i: (-lengths[i], i))
    heap = [(0, r) for r in range(world_size)]
    heapq.heapify(heap)
    parts: list[list[int]] = [[] for _ in range(world_size)]
    for i in order:
        load, r = heapq.heappop(heap)
        parts[r].append(i)
        heapq.heappush(heap, (load + lengths[i], r))
    return [sorted(p) for p in parts]


def local_rows(cu_seqlens, seq_ids):
    """Packed rows and local cu_seqlens of the given sequences.

    Returns (rows, cu_local): `rows` indexes the token-major arrays of the full
    batch, `cu_local` is the int32 cu_seqlens of the rank's packed batch.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = [int(cu[i + 1] - cu[i]) for i in seq_ids]
    rows = (np.concatenate([np.arange(cu[i], cu[i + 1]) for i in seq_ids])
            if seq_ids else np.zeros(0, dtype=np.int64))
    cu_local = np.zeros(len(seq_ids) + 1, dtype=np.int32)
    cu_local[1:] = np.cumsum(lens)
    return rows.astype(np.int64), cu_local


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank scalar over the default process group (or the value
    itself when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
