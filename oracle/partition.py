"""Oracle for the partitions of a packed multi-ragged batch.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "DanLing NestedTensor: Composable Multi-Ragged Tensors for Deep
Learning":
  * section 3.1 "Numerical storage", Eq. 2: sample i occupies packed rows
    [o_i, o_{i+1}) with p_i the product of its ragged extents, o_i = sum_{k<i} p_k
    and T = sum_i p_i.  For singles p_i = N_i; for square pairs p_i = N_i^2.
  * section 3.2, Eq. 3: the packed row of ragged coordinates (a, b) in sample i
    is l_i(a, b) = o_i + a * N_i + b.
  * Figure 2 and section 3.2 "Creating axes through broadcasting": for lengths
    (2, 3) the sample offsets go from [0, 2, 5] (singles) to [0, 4, 13]
    (pairs); the second-level splits delimit each pair row's cells.
  * Appendix A "Structural invariants": o_0 = 0, o_{i+1} - o_i = p_i, o_B = T;
    the innermost splits of a pair tensor hold 1 + sum_i N_i entries.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Sequence

import numpy as np


@dataclass
class Partition:
    lengths: np.ndarray     # N_i, int64 (B,)
    cu_seqlens: np.ndarray  # single offsets eta (Eq. 4) = o for singles, (B+1,)
    pair_off: np.ndarray    # o for square pairs, (B+1,)
    row_start: np.ndarray   # second-level splits: first cell of each pair row, (T+1,)
    row_sample: np.ndarray  # sample owning each pair row, (T,)
    T: int                  # sum N_i
    P: int                  # sum N_i^2
    max_len: int


def sample_offsets(p: Sequence[int]) -> np.ndarray:
    """o_0 = 0 and o_{i+1} = o_i + p_i (Eq. 2), written out as a loop."""
    o = [0]
    for pi in p:
        o.append(o[-1] + int(pi))
    return np.asarray(o, dtype=np.int64)


def packed_pair_row(pair_off: np.ndarray, lengths: np.ndarray, i: int, a: int, b: int) -> int:
    """l_i(a, b) = o_i + a * N_i + b (Eq. 3 with q = 2, n_{i,r_2} = N_i)."""
    return int(pair_off[i]) + a * int(lengths[i]) + b


def partition(lengths: Sequence[int]) -> Partition:
    N = [int(n) for n in lengths]
    if any(n < 0 for n in N):
        raise ValueError("lengths must be non-negative")
    N_arr = np.asarray(N, dtype=np.int64)
    cu = sample_offsets(N)                       # p_i = N_i (singles)
    pair_off = sample_offsets([n * n for n in N])  # p_i = N_i^2 (square pairs)
    row_start = []
    row_sample = []
    for i, n in enumerate(N):
        for a in range(n):
            row_start.append(packed_pair_row(pair_off, N_arr, i, a, 0))
            row_sample.append(i)
    row_start.append(int(pair_off[-1]))
    return Partition(
        lengths=N_arr, cu_seqlens=cu, pair_off=pair_off,
        row_start=np.asarray(row_start, dtype=np.int64),
        row_sample=np.asarray(row_sample, dtype=np.int64),
        T=int(cu[-1]), P=int(pair_off[-1]), max_len=max(N) if N else 0)


def padded_cells(lengths: Sequence[int]) -> int:
    """Cells of the padded envelope B * N_max^2 (abstract; section 1)."""
    N = [int(n) for n in lengths]
    return len(N) * (max(N) if N else 0) ** 2
