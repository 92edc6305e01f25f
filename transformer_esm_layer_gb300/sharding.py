"""Splitting a packed batch across GPUs.

The sequences of a packed batch never interact (each attends only to itself), so a
multi-GPU forward is a set of independent replicas, each encoding its own share of the
sequences: no collective is needed on the data path.  The split balances work, not
tokens: a sequence of length L costs 2 L (4 d^2 + 2 d f) GEMM FLOPs plus 4 d L^2 attention
FLOPs per layer.  Longest-first greedy assignment to the least-loaded rank is the
sort-then-bucket idea of the length-aware sampler in section 5.2 of the hotelren.com guide.

Training adds one exchange: the parameters are shared by every sequence and the gradient of
a packed batch is the sum of its sequences' gradients, so ranks that each backpropagated
their own share hold partial sums, and one all-reduce (sum) of the gradients gives every
rank the batch gradient (data parallelism of the hotelren.com guide's training loop).

The masked-LM loss is a mean over the scored tokens of the whole batch, so its normaliser
is global: a data-parallel step first sums the ranks' scored counts (``global_scored_count``)
and passes that count to the loss backward (``EsmEncoder.lm_head_backward(...,
loss_count=...)``); each rank then differentiates its share of the same loss, and the
all-reduce of the gradients gives the batch gradient.  With each rank's own count instead,
the sum would be the sum of the ranks' means, wrong by about the world size.
"""
from __future__ import annotations

import heapq
from typing import List, Optional, Sequence, Tuple

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


def allreduce_gradients(tensors: Sequence, group=None, bucket_bytes: int = 256 << 20) -> int:
    """Sum the gradient tensors over the ranks of the process group, in place.

    Every rank passes tensors of the same shapes, dtypes and order.  They are packed in that
    order into flat buckets of at most bucket_bytes (a tensor larger than that is a bucket on
    its own) and each bucket is one all-reduce, so the collective sequence is identical on
    every rank.  Returns the number of bytes reduced per rank."""
    import torch
    import torch.distributed as dist

    total = 0
    bucket: List = []
    size = 0

    def flush(b: List) -> None:
        if not b:
            return
        flat = torch.cat([t.reshape(-1) for t in b])
        dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
        off = 0
        for t in b:
            n = t.numel()
            t.copy_(flat[off:off + n].view_as(t))
            off += n

    for t in tensors:
        nbytes = t.numel() * t.element_size()
        total += nbytes
        if bucket and (size + nbytes > bucket_bytes or t.dtype != bucket[0].dtype or t.device != bucket[0].device):
            flush(bucket)
            bucket, size = [], 0
        bucket.append(t)
        size += nbytes
    flush(bucket)
    return total


def global_scored_count(targets, group=None, ignore_index: int = -100):
    """Number of scored masked-LM targets over all ranks (an all-reduce sum of each rank's
    count): the normaliser of the batch's mean loss.  ``targets`` is this rank's int tensor
    (any device the process group serves); returns an int32 tensor of one element on the
    same device, ready to pass as ``loss_count``."""
    import torch
    import torch.distributed as dist

    n = (targets != ignore_index).sum().to(torch.int64).reshape(1)
    dist.all_reduce(n, op=dist.ReduceOp.SUM, group=group)
    return n.to(torch.int32)
