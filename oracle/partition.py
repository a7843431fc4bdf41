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
  * section 3.2 "Consuming one logical axis", Eq. 4: a rectangular pair state
    P_i of N_i x M_i cells packs cell (a, b) at o_i + a * M_i + b, with o the
    exclusive scan of N_i * M_i, and its rows are grouped by
    eta_i = sum_{k<i} N_k.
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


@dataclass
class RectPartition:
    rows: np.ndarray        # N_i, int64 (B,)
    cols: np.ndarray        # M_i, int64 (B,)
    cu_rows: np.ndarray     # eta of Eq. 4: offsets of the row singles, (B+1,)
    cu_cols: np.ndarray     # offsets of the column singles, (B+1,)
    pair_off: np.ndarray    # o: exclusive scan of N_i * M_i, (B+1,)
    row_start: np.ndarray   # first cell of each pair row, (T_rows+1,)
    row_sample: np.ndarray  # sample owning each pair row, (T_rows,)
    T_rows: int
    T_cols: int
    P: int
    max_rows: int
    max_cols: int


def packed_rect_row(pair_off: np.ndarray, cols: np.ndarray, i: int, a: int, b: int) -> int:
    """o_i + a * M_i + b (the packed row of cell (a, b) in Eq. 4)."""
    return int(pair_off[i]) + a * int(cols[i]) + b


def partition_rect(rows: Sequence[int], cols: Sequence[int]) -> RectPartition:
    """Partitions of a batch of rectangular pair states: row singles of
    lengths N_i, column singles of lengths M_i, N_i x M_i cells each."""
    N = [int(n) for n in rows]
    M = [int(m) for m in cols]
    if len(N) != len(M):
        raise ValueError("one column length per sample")
    if any(n < 0 for n in N) or any(m < 0 for m in M):
        raise ValueError("lengths must be non-negative")
    M_arr = np.asarray(M, dtype=np.int64)
    cu_r = sample_offsets(N)
    cu_c = sample_offsets(M)
    pair_off = sample_offsets([n * m for n, m in zip(N, M)])
    row_start, row_sample = [], []
    for i, n in enumerate(N):
        for a in range(n):
            row_start.append(packed_rect_row(pair_off, M_arr, i, a, 0))
            row_sample.append(i)
    row_start.append(int(pair_off[-1]))
    return RectPartition(
        rows=np.asarray(N, dtype=np.int64), cols=M_arr, cu_rows=cu_r, cu_cols=cu_c, pair_off=pair_off,
        row_start=np.asarray(row_start, dtype=np.int64), row_sample=np.asarray(row_sample, dtype=np.int64),
        T_rows=int(cu_r[-1]), T_cols=int(cu_c[-1]), P=int(pair_off[-1]),
        max_rows=max(N) if N else 0, max_cols=max(M) if M else 0)


def padded_cells(lengths: Sequence[int]) -> int:
    """Cells of the padded envelope B * N_max^2 (abstract; section 1)."""
    N = [int(n) for n in lengths]
    return len(N) * (max(N) if N else 0) ** 2
