"""Splitting a packed batch across ranks.

Every step of the block and of varlen attention is sample-local ("DanLing
NestedTensor", Appendix A, reference semantics: sample-local operations equal
independent per-element computations), so a batch shards by sample with no
exchange in the forward pass: each rank builds its own partition over its
own samples.  The pair work of sample i grows as N_i^2 (attention: n_i^2),
so samples are placed longest-processing-time first: sorted by N_i^2,
descending, each onto the rank with the least work so far.
"""
from __future__ import annotations

from typing import List, Sequence


def shard_samples(lengths: Sequence[int], world: int) -> List[List[int]]:
    """Sample indices per rank (each list ascending), balanced by N_i^2."""
    if world < 1:
        raise ValueError("world must be >= 1")
    load = [0] * world
    shards: List[List[int]] = [[] for _ in range(world)]
    order = sorted(range(len(lengths)), key=lambda i: (-int(lengths[i]) ** 2, i))
    for i in order:
        r = min(range(world), key=lambda k: (load[k], k))
        shards[r].append(i)
        load[r] += int(lengths[i]) ** 2
    return [sorted(s) for s in shards]


def shard_rows(lengths: Sequence[int], samples: Sequence[int]) -> List[int]:
    """Packed single rows (indices into the whole batch) of the given samples,
    in the samples' order."""
    starts = [0]
    for n in lengths:
        starts.append(starts[-1] + int(n))
    rows: List[int] = []
    for i in samples:
        rows.extend(range(starts[i], starts[i + 1]))
    return rows
