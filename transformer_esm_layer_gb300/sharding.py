"""Splitting a packed batch across GPUs.

The sequences of a packed batch never interact (each attends only to itself), so a
multi-GPU forward is a set of independent replicas, each encoding its own share of the
sequences: no collective is needed on the data path.  The split balances work, not
tokens: a sequence of length L costs 2 L (4 d^2 + 2 d f) GEMM FLOPs plus 4 d L^2 attention
FLOPs per layer.  Longest-first greedy assignment to the least-loaded rank is the
sort-then-bucket idea of the length-aware sampler in section 5.2 of the hotelren.com guide.
"""
from __future__ import annotations

import heapq
from typing import List, Sequence, Tuple

import numpy as np


def sequence_cost(L: int, hidden: int, ffn: int) -> float:
    """Per-layer FLOPs of one sequence of length L."""
    return 2.0 * L * (4 * hidden * hidden + 2 * hidden * ffn) + 4.0 * hidden * float(L) * float(L)


def shard_by_work(lengths: Sequence[int], world: int, hidden: int, ffn: int) -> List[List[int]]:
    """Indices of the sequences each rank encodes (each list in batch order).

    Longest-first greedy: every sequence goes to the rank with the least work so far (ties
    to the lowest rank), which keeps the max/mean work ratio within one sequence's cost."""
    if world <= 0:
        raise ValueError("world must be positive")
    order = sorted(range(len(lengths)), key=lambda i: (-int(lengths[i]), i))
    heap = [(0.0, r) for r in range(world)]
    out: List[List[int]] = [[] for _ in range(world)]
    for i in order:
        load, r = heapq.heappop(heap)
        out[r].append(i)
        heapq.heappush(heap, (load + sequence_cost(int(lengths[i]), hidden, ffn), r))
    return [sorted(s) for s in out]


def local_batch(tokens: np.ndarray, lengths: Sequence[int], indices: Sequence[int]) -> Tuple[np.ndarray, List[int]]:
    """The packed tokens and lengths of the chosen sequences (in the given order)."""
    cu = np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))])
    parts = [tokens[cu[i]:cu[i + 1]] for i in indices]
    toks = np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)
    return toks, [int(lengths[i]) for i in indices]
