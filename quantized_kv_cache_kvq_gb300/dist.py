"""Multi-GPU host logic: sequences are independent units, so ranks shard them with no data-path collective.

WitCert §6.3.10 runs the meter under tensor parallelism without describing a
cross-rank exchange, and leaves a cross-rank gate unverified; the decode path
itself needs none: every (sequence, kv head) unit is attended on one GPU.  The
only cross-rank quantities are the tiny meter summaries (coverage counts,
non-finite counts), reduced on the host after the step.

- ``shard_sequences``: split a batch across ranks, balancing attended tokens.
- ``reduce_meter_counts``: sum the four ``kvq_meter`` counters over ranks
  (an all-reduce on CPU tensors; gloo in the tests, any backend in use).
"""
from __future__ import annotations

import numpy as np

__all__ = ["shard_sequences", "reduce_meter_counts"]


def shard_sequences(seq_lens, world_size: int, prefix_len: int = 0) -> list[np.ndarray]:
    """Assign every sequence to one rank so that the attended tokens per rank are balanced.

    Greedy longest-first onto the least-loaded rank (ties to the lower rank);
    returns, per rank, the sorted indices of its sequences.  Deterministic.
    """
    lens = np.asarray(seq_lens, dtype=np.int64)
    if world_size <= 0:
        raise ValueError("world_size must be positive")
    cost = lens + int(prefix_len)
    order = sorted(range(len(lens)), key=lambda i: (-int(cost[i]), i))
    load = [0] * world_size
    out: list[list[int]] = [[] for _ in range(world_size)]
    for i in order:
        r = min(range(world_size), key=lambda k: (load[k], k))
        out[r].append(i)
        load[r] += int(cost[i])
    return [np.array(sorted(o), dtype=np.int64) for o in out]


def reduce_meter_counts(counts, group=None):
    """Sum per-rank meter counters [covered_A, covered_B, nonfinite, cells] over the process group."""
    import torch
    import torch.distributed as dist

    t = torch.as_tensor(counts, dtype=torch.int64).cpu().clone()
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return t
