"""Oracle for the single->pair->single block.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "DanLing NestedTensor: Composable Multi-Ragged Tensors for Deep
Learning", section 3, Eq. 1, for a sample X_i of shape (N_i, C):

    P_i[a, b]   = u(X_i[a]) + v(X_i[b])
    P~_i        = P_i + h(LN_{C_p}(P_i))
    X~_i[a]     = X_i[a] + g( (1/N_i) * sum_b P~_i[a, b] )

with u, v projections to pair width C_p (Appendix A.1: the pair is the plain
sum of the two projections, no activation at construction), g mapping back to
width C, and projections computed as V W^T + b (section 3.3, "Dense work
across valid positions").  Readings where the pages leave a step open:

* h is a ReLU MLP  C_p -> H_t -> C_p  (the paper's measured h is SwiGLU; the
  block built here is the LayerNorm -> Linear -> ReLU -> Linear transition).
* u and v carry no bias; transition and g biases are optional.
* LN_{C_p} normalises the C_p features of one cell with the biased variance
  (divide by C_p), eps added to the variance, then gamma * x + beta.
* The mean runs over the column index b for each row a (Eq. 1's sum over b,
  and Eq. 4's grouping of cells with "the same sample and row coordinate").

Packing follows Eq. 2/3: cell (a, b) of sample i is packed row
o_i + a * N_i + b with o the exclusive scan of N_i^2.

Rectangular pairs (section 3.2 "Consuming one logical axis", Eq. 4;
Appendix A.1 "the rectangular variant has distinct row and column inputs and
divides its column mean by M_i"): rows come from X_i (N_i x C), columns from
Z_i (M_i x C), P_i[a, b] = u(X_i[a]) + v(Z_i[b]) over N_i x M_i cells packed
at o_i + a * M_i + b, and the mean over b divides by M_i.  Reading: a sample
with M_i = 0 has an empty column sum; its row means are taken as zero (the
pages define the mean for non-empty rows only).

SwiGLU transition (Eq. 1: h is "a SwiGLU feature update" after Shazeer 2020;
Appendix A.1: transition expansion four): h(y) = W2 (SiLU(W1 y + b1) *
(W3 y + b3)) + b2 with SiLU(x) = x sigmoid(x) (Swish with beta = 1), W1 the
gate and W3 the value projection, both C_p -> H_t.  Biases are optional.

Everything is float64; inputs are the exact values handed to the GPU.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

from .partition import packed_rect_row, partition, partition_rect


def linear(x: np.ndarray, W: np.ndarray, b: Optional[np.ndarray] = None) -> np.ndarray:
    """x W^T + b, with W stored (out_features, in_features)."""
    y = x @ W.T
    if b is not None:
        y = y + b
    return y


def layer_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis: biased variance, eps inside the root."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * gamma + beta


def h_theta(x, W1, b1, W2, b2):
    """Feature update: Linear(C_p -> H_t), ReLU, Linear(H_t -> C_p)."""
    return linear(np.maximum(linear(x, W1, b1), 0.0), W2, b2)


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x) = x / (1 + exp(-x))."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def h_swiglu(x, W1, b1, W3, b3, W2, b2):
    """Gated update: Linear(C_p -> H_t) through SiLU, times a second
    Linear(C_p -> H_t), then Linear(H_t -> C_p)."""
    return linear(silu(linear(x, W1, b1)) * linear(x, W3, b3), W2, b2)


def transition_swiglu(P, gamma, beta, eps, W1, b1, W3, b3, W2, b2):
    """P~ = P + h_swiglu(LN(P)) on every cell independently."""
    return P + h_swiglu(layer_norm(P, gamma, beta, eps), W1, b1, W3, b3, W2, b2)


def transition(P, gamma, beta, eps, W1, b1, W2, b2):
    """P~ = P + h(LN(P)) on every cell independently (Eq. 1, second line)."""
    return P + h_theta(layer_norm(P, gamma, beta, eps), W1, b1, W2, b2)


@dataclass
class Weights:
    """float64 copies of one block's parameters, layout (out, in)."""
    W_a: np.ndarray
    W_b: np.ndarray
    gamma: np.ndarray
    beta: np.ndarray
    eps: float
    W1: np.ndarray
    b1: Optional[np.ndarray]
    W2: np.ndarray
    b2: Optional[np.ndarray]
    W_g: np.ndarray
    b_g: Optional[np.ndarray]


@dataclass
class SampleResult:
    P: np.ndarray        # (N, N, C_p) pair state before the transition
    P_tilde: np.ndarray  # (N, N, C_p)
    M: np.ndarray        # (N, C_p) row means of P~
    X_tilde: np.ndarray  # (N, C)


def block_sample(X: np.ndarray, w: Weights, X_right: Optional[np.ndarray] = None) -> SampleResult:
    """Eq. 1 for one sample, densely.  ``X_right`` (default X) feeds v."""
    Xr = X if X_right is None else X_right
    U = linear(X, w.W_a)                       # u(X[a])
    V = linear(Xr, w.W_b)                      # v(X[b])
    P = U[:, None, :] + V[None, :, :]          # P[a, b] = u(X[a]) + v(X[b])
    P_tilde = transition(P, w.gamma, w.beta, w.eps, w.W1, w.b1, w.W2, w.b2)
    N = X.shape[0]
    M = P_tilde.sum(axis=1) / N                # (1/N) sum_b P~[a, b]
    X_tilde = X + linear(M, w.W_g, w.b_g)
    return SampleResult(P, P_tilde, M, X_tilde)


def block_sample_rect(X: np.ndarray, Z: np.ndarray, w: Weights) -> SampleResult:
    """The rectangular block for one sample: rows from X (N x C), columns
    from Z (M x C), mean over the M columns."""
    U = linear(X, w.W_a)                       # u(X[a]), (N, C_p)
    V = linear(Z, w.W_b)                       # v(Z[b]), (M, C_p)
    P = U[:, None, :] + V[None, :, :]          # (N, M, C_p)
    P_tilde = transition(P, w.gamma, w.beta, w.eps, w.W1, w.b1, w.W2, w.b2)
    Mi = Z.shape[0]
    Mean = P_tilde.sum(axis=1) / Mi if Mi > 0 else np.zeros((X.shape[0], U.shape[1]))
    X_tilde = X + linear(Mean, w.W_g, w.b_g)
    return SampleResult(P, P_tilde, Mean, X_tilde)


@dataclass
class PackedResult:
    z: np.ndarray        # (P, C_p) packed pair state before the transition
    z_tilde: np.ndarray  # (P, C_p) packed P~
    m: np.ndarray        # (T, C_p) packed row means
    s_out: np.ndarray    # (T, C) packed X~


def block_packed(lengths: Sequence[int], s: np.ndarray, w: Weights) -> PackedResult:
    """Run ``block_sample`` on every sample and pack the results by Eq. 2/3."""
    part = partition(lengths)
    C_p = w.W_a.shape[0]
    z = np.zeros((part.P, C_p))
    z_tilde = np.zeros((part.P, C_p))
    m = np.zeros((part.T, C_p))
    s_out = np.zeros((part.T, s.shape[1]))
    for i, N in enumerate(part.lengths):
        N = int(N)
        if N == 0:
            continue
        X = s[part.cu_seqlens[i]:part.cu_seqlens[i + 1]]
        r = block_sample(X, w)
        o = int(part.pair_off[i])
        z[o:o + N * N] = r.P.reshape(N * N, C_p)
        z_tilde[o:o + N * N] = r.P_tilde.reshape(N * N, C_p)
        m[part.cu_seqlens[i]:part.cu_seqlens[i + 1]] = r.M
        s_out[part.cu_seqlens[i]:part.cu_seqlens[i + 1]] = r.X_tilde
    return PackedResult(z, z_tilde, m, s_out)


def block_packed_rect(rows: Sequence[int], cols: Sequence[int], s_row: np.ndarray, s_col: np.ndarray,
                      w: Weights) -> PackedResult:
    """``block_sample_rect`` on every sample, packed by Eq. 4's layout."""
    part = partition_rect(rows, cols)
    C_p = w.W_a.shape[0]
    z = np.zeros((part.P, C_p))
    z_tilde = np.zeros((part.P, C_p))
    m = np.zeros((part.T_rows, C_p))
    s_out = np.zeros((part.T_rows, s_row.shape[1]))
    for i in range(len(part.rows)):
        N, M = int(part.rows[i]), int(part.cols[i])
        if N == 0:
            continue
        X = s_row[part.cu_rows[i]:part.cu_rows[i + 1]]
        Z = s_col[part.cu_cols[i]:part.cu_cols[i + 1]]
        r = block_sample_rect(X, Z, w)
        o = int(part.pair_off[i])
        z[o:o + N * M] = r.P.reshape(N * M, C_p)
        z_tilde[o:o + N * M] = r.P_tilde.reshape(N * M, C_p)
        m[part.cu_rows[i]:part.cu_rows[i + 1]] = r.M
        s_out[part.cu_rows[i]:part.cu_rows[i + 1]] = r.X_tilde
    return PackedResult(z, z_tilde, m, s_out)


def block_padded_gathered(lengths: Sequence[int], s: np.ndarray, w: Weights) -> PackedResult:
    """Same block through the padded envelope: pad every sample to N_max with
    zero rows, compute all B x N_max x N_max cells, take the row mean over the
    valid columns only (divide by N_i), then gather the valid cells in packed
    order.  Shares no indexing with ``block_packed``."""
    N = [int(n) for n in lengths]
    B, N_max, C = len(N), max(N) if N else 0, s.shape[1]
    C_p = w.W_a.shape[0]
    X_pad = np.zeros((B, N_max, C))
    valid = np.zeros((B, N_max), dtype=bool)
    start = 0
    for i, n in enumerate(N):
        X_pad[i, :n] = s[start:start + n]
        valid[i, :n] = True
        start += n
    U = linear(X_pad, w.W_a)
    V = linear(X_pad, w.W_b)
    P = U[:, :, None, :] + V[:, None, :, :]                    # (B, Nm, Nm, C_p)
    P_tilde = transition(P, w.gamma, w.beta, w.eps, w.W1, w.b1, w.W2, w.b2)
    col_mask = valid[:, None, :, None]                         # valid b
    counts = np.maximum(np.asarray(N, dtype=np.float64), 1.0)[:, None, None]
    M = np.where(col_mask, P_tilde, 0.0).sum(axis=2) / counts  # (B, Nm, C_p)
    X_tilde = X_pad + linear(M, w.W_g, w.b_g)
    pair_mask = valid[:, :, None] & valid[:, None, :]
    return PackedResult(z=P[pair_mask], z_tilde=P_tilde[pair_mask],
                        m=M[valid], s_out=X_tilde[valid])


# ----------------------------------------------------------------------------
# The block split at the library's call boundaries.  Each function takes the
# packed tensors a call takes and computes its output one sample at a time.
# ----------------------------------------------------------------------------

def pair_broadcast(lengths, s_left, s_right, W_a, W_b) -> np.ndarray:
    """z[l_i(a, b)] = u(X_L,i[a]) + v(X_R,i[b]) over the sum N_i^2 cells,
    one sample at a time (dense N_i x N_i block, then packed by Eq. 3)."""
    part = partition(lengths)
    C_p = W_a.shape[0]
    z = np.zeros((part.P, C_p))
    for i, N in enumerate(part.lengths):
        N = int(N)
        if N == 0:
            continue
        sl = slice(part.cu_seqlens[i], part.cu_seqlens[i + 1])
        U = linear(s_left[sl], W_a)
        V = linear(s_right[sl], W_b)
        o = int(part.pair_off[i])
        z[o:o + N * N] = (U[:, None, :] + V[None, :, :]).reshape(N * N, C_p)
    return z


def pair_transition(z, gamma, beta, eps, W1, b1, W2, b2) -> np.ndarray:
    """Row-wise z + h(LN(z)); the transition retains the partitions
    (section 3.2 "Retaining structure through feature transformations")."""
    return transition(z, gamma, beta, eps, W1, b1, W2, b2)


def pair_reduce(lengths, z, W_g=None, b_g=None, s_in=None):
    """Eq. 4 with M_i = N_i, divided by N_i (the square-pair mean of Eq. 1):
        m[eta_i + a] = (1/N_i) sum_b z[o_i + a N_i + b]
    then, when W_g is given, s_out = s_in + m W_g^T + b_g (s_in optional)."""
    part = partition(lengths)
    C_p = z.shape[1]
    m = np.zeros((part.T, C_p))
    for i, N in enumerate(part.lengths):
        N = int(N)
        if N == 0:
            continue
        o = int(part.pair_off[i])
        cells = z[o:o + N * N].reshape(N, N, C_p)          # [a, b, :]
        m[part.cu_seqlens[i]:part.cu_seqlens[i + 1]] = cells.sum(axis=1) / N
    if W_g is None:
        return m, None
    s_out = linear(m, W_g, b_g)
    if s_in is not None:
        s_out = s_in + s_out
    return m, s_out


def pair_broadcast_rect(rows, cols, s_row, s_col, W_a, W_b) -> np.ndarray:
    """z[o_i + a M_i + b] = u(X_i[a]) + v(Z_i[b]) over the sum N_i M_i cells."""
    part = partition_rect(rows, cols)
    z = np.zeros((part.P, W_a.shape[0]))
    for i in range(len(part.rows)):
        N, M = int(part.rows[i]), int(part.cols[i])
        U = linear(s_row[part.cu_rows[i]:part.cu_rows[i + 1]], W_a)
        V = linear(s_col[part.cu_cols[i]:part.cu_cols[i + 1]], W_b)
        for a in range(N):
            for b in range(M):
                z[packed_rect_row(part.pair_off, part.cols, i, a, b)] = U[a] + V[b]
    return z


def pair_reduce_rect(rows, cols, z, W_g=None, b_g=None, s_in=None):
    """Eq. 4's column sum divided by M_i: m[eta_i + a] = (1/M_i) sum_b
    z[o_i + a M_i + b] (zero when M_i = 0); optionally s_out = s_in + g(m)."""
    part = partition_rect(rows, cols)
    m = np.zeros((part.T_rows, z.shape[1]))
    for i in range(len(part.rows)):
        N, M = int(part.rows[i]), int(part.cols[i])
        for a in range(N):
            if M == 0:
                continue
            acc = np.zeros(z.shape[1])
            for b in range(M):
                acc += z[packed_rect_row(part.pair_off, part.cols, i, a, b)]
            m[part.cu_rows[i] + a] = acc / M
    s_out = None if W_g is None else s_in + linear(m, W_g, b_g)
    return m, s_out


def stacked_blocks(lengths, s, weights: List[Weights]):
    """Blocks chained through the singles: block k+1 takes X~ of block k and
    builds a fresh pair state (Eq. 1 takes only X).  Returns the final singles
    and the last block's packed results."""
    x = s
    last = None
    for w in weights:
        last = block_packed(lengths, x, w)
        x = last.s_out
    return x, last


# ----------------------------------------------------------------------------
# Sampled evaluation for full-size checks: a few cells / rows computed one by
# one from their definition, without forming the whole pair state.
# ----------------------------------------------------------------------------

def block_cells(lengths, s, w: Weights, cells: Sequence[int]):
    """P and P~ at the listed packed cells.  Cell c belongs to the sample i
    with o_i <= c < o_{i+1}; its coordinates are a = (c - o_i) // N_i and
    b = (c - o_i) % N_i (Eq. 3 inverted)."""
    part = partition(lengths)
    cells = np.asarray(cells, dtype=np.int64)
    i = np.searchsorted(part.pair_off, cells, side="right") - 1
    N = part.lengths[i]
    a = (cells - part.pair_off[i]) // N
    b = (cells - part.pair_off[i]) % N
    ra = part.cu_seqlens[i] + a
    rb = part.cu_seqlens[i] + b
    P = linear(s[ra], w.W_a) + linear(s[rb], w.W_b)
    return P, transition(P, w.gamma, w.beta, w.eps, w.W1, w.b1, w.W2, w.b2)


def block_rows(lengths, s, w: Weights, rows: Sequence[int]):
    """m and X~ at the listed packed single rows: the whole pair row a of its
    sample is formed and reduced (Eq. 1, third line)."""
    part = partition(lengths)
    rows = np.asarray(rows, dtype=np.int64)
    m = np.zeros((len(rows), w.W_a.shape[0]))
    for k, r in enumerate(rows):
        i = int(np.searchsorted(part.cu_seqlens, r, side="right") - 1)
        lo, hi = int(part.cu_seqlens[i]), int(part.cu_seqlens[i + 1])
        P_row = linear(s[r], w.W_a)[None, :] + linear(s[lo:hi], w.W_b)   # P[a, b] over b
        P_t = transition(P_row, w.gamma, w.beta, w.eps, w.W1, w.b1, w.W2, w.b2)
        m[k] = P_t.sum(axis=0) / (hi - lo)
    return m, s[rows] + linear(m, w.W_g, w.b_g)
