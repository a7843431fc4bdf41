"""Oracle for variable-length (cu_seqlens) softmax attention.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "Variable-length attention and data packing":
  * "What it is": the packed batch is one concatenated sequence plus
    cu_seqlens, and attention is computed only within each real sequence;
  * "How it works": query rows of a sequence see only that sequence's keys,
    so the cost is the sum of per-sequence len^2 terms;
  * "Core math" (C): a block-diagonal mask seg[i] == seg[j] applied to the
    scores with -inf off the diagonal blocks gives zero cross-sample mass and
    rows that still sum to one.
"DanLing NestedTensor", section 3.3 "Attention through packed blocks": the
output adopts the query structure (token-major, static head and feature axes).

Readings: non-causal by default; scale passed in (d^-1/2 by default); the
log-sum-exp is natural-log, lse[h, t] = log sum_k exp(scale * q_t . k_k) over
t's segment.  Cross-attention ("DanLing NestedTensor" section 3.3: the output
adopts the query structure, query and key lengths may differ) takes separate
query and key offsets.  Causal masking ("Variable-length attention and data
packing", "How to use it": the varlen call of its template sets the causal
flag) is aligned to the bottom-right corner when the lengths differ: query i of a
segment with n_q queries and n_k keys sees keys j <= i + (n_k - n_q); a query
that sees no key returns zeros with lse = -inf.

Backward (the gradients of the same per-segment attention with respect to
q, k and v for an upstream gradient dO), written from the chain rule of
softmax(scale Q K^T) V: with P the attention matrix of a segment,
dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dO * O)), dQ = scale dS K,
dK = scale dS^T Q; masked entries have P = 0 and get no gradient.
"""
from __future__ import annotations

from typing import Optional, Sequence, Tuple

import numpy as np


def _softmax_rows(S: np.ndarray) -> np.ndarray:
    S = S - S.max(axis=-1, keepdims=True)
    E = np.exp(S)
    return E / E.sum(axis=-1, keepdims=True)


def segment_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool = False):
    """Dense attention of one segment: q is (n_q, H, d), k and v (n_k, H, d).
    Returns O (n_q, H, d) and lse (H, n_q)."""
    nq, H, d = q.shape
    nk = k.shape[0]
    O = np.zeros((nq, H, v.shape[2]))
    lse = np.full((H, nq), -np.inf)
    allowed = np.ones((nq, nk), dtype=bool)
    if causal:
        allowed = np.arange(nk)[None, :] <= np.arange(nq)[:, None] + (nk - nq)
    for h in range(H):
        S = (q[:, h, :] @ k[:, h, :].T) * scale            # (n_q, n_k) explicit scores
        for i in range(nq):
            if not allowed[i].any():
                continue                                     # no key: zeros, lse = -inf
            s = S[i, allowed[i]]
            mx = s.max()
            e = np.exp(s - mx)
            O[i, h, :] = (e / e.sum()) @ v[allowed[i], h, :]
            lse[h, i] = mx + np.log(e.sum())
    return O, lse


def varlen_attention(q, k, v, cu_seqlens: Sequence[int], scale: Optional[float] = None,
                     segments: Optional[Sequence[int]] = None, causal: bool = False,
                     cu_seqlens_k: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Attention restricted to each segment, one segment at a time: queries
    [cu[b], cu[b+1]) against keys [cu_k[b], cu_k[b+1]) (cu_k = cu for
    self-attention).  ``segments`` limits the work to the listed segment
    indices (the other rows of O and lse stay zero)."""
    T, H, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    cu_k = cu_seqlens if cu_seqlens_k is None else cu_seqlens_k
    O = np.zeros((T, H, v.shape[2]))
    lse = np.zeros((H, T))
    B = len(cu_seqlens) - 1
    for b in (range(B) if segments is None else segments):
        lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        klo, khi = int(cu_k[b]), int(cu_k[b + 1])
        if hi == lo:
            continue
        O[lo:hi], lse[:, lo:hi] = segment_attention(q[lo:hi], k[klo:khi], v[klo:khi], scale, causal)
    return O, lse


def segment_attention_backward(q, k, v, do, scale: float, causal: bool = False):
    """Gradients of one segment's attention: q, do (n_q, H, d); k, v (n_k, H, d).
    Returns dq, dk, dv with the shapes of q, k, v."""
    nq, H, d = q.shape
    nk = k.shape[0]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    allowed = np.ones((nq, nk), dtype=bool)
    if causal:
        allowed = np.arange(nk)[None, :] <= np.arange(nq)[:, None] + (nk - nq)
    for h in range(H):
        S = (q[:, h, :] @ k[:, h, :].T) * scale
        S = np.where(allowed, S, -np.inf)
        P = np.zeros_like(S)
        for i in range(nq):
            if allowed[i].any():
                e = np.exp(S[i] - S[i][allowed[i]].max())
                P[i] = e / e.sum()
        O = P @ v[:, h, :]
        dO = do[:, h, :]
        dv[:, h, :] = P.T @ dO
        dP = dO @ v[:, h, :].T
        Drow = (dO * O).sum(axis=1, keepdims=True)
        dS = P * (dP - Drow)
        dq[:, h, :] = scale * dS @ k[:, h, :]
        dk[:, h, :] = scale * dS.T @ q[:, h, :]
    return dq, dk, dv


def varlen_attention_backward(q, k, v, do, cu_seqlens, scale: Optional[float] = None, causal: bool = False,
                              cu_seqlens_k=None, segments: Optional[Sequence[int]] = None):
    """Gradients of ``varlen_attention`` segment by segment; ``segments``
    limits the work to the listed segments (the other rows stay zero)."""
    T, H, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    cu_k = cu_seqlens if cu_seqlens_k is None else cu_seqlens_k
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    B = len(cu_seqlens) - 1
    for b in (range(B) if segments is None else segments):
        lo, hi = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        klo, khi = int(cu_k[b]), int(cu_k[b + 1])
        if hi == lo or khi == klo:
            continue
        dq[lo:hi], dk[klo:khi], dv[klo:khi] = segment_attention_backward(q[lo:hi], k[klo:khi], v[klo:khi],
                                                                         do[lo:hi], scale, causal)
    return dq, dk, dv


def masked_full_attention(q, k, v, seg_ids: Sequence[int], scale: Optional[float] = None):
    """Full T x T attention with scores set to -inf wherever
    seg[i] != seg[j] ("Core math" (C)).  Tiny inputs only.  Returns O and the
    attention matrices A (H, T, T)."""
    T, H, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    seg = np.asarray(seg_ids)
    block = seg[:, None] == seg[None, :]
    O = np.zeros((T, H, v.shape[2]))
    A_all = np.zeros((H, T, T))
    for h in range(H):
        S = (q[:, h, :] @ k[:, h, :].T) * scale
        A = _softmax_rows(np.where(block, S, -np.inf))
        A_all[h] = A
        O[:, h, :] = A @ v[:, h, :]
    return O, A_all


def masked_full_attention_causal(q, k, v, seg_ids: Sequence[int], scale: Optional[float] = None):
    """Full T x T attention with the block-diagonal mask and, within a block,
    keys after the query masked too (self-attention, equal lengths)."""
    T, H, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    seg = np.asarray(seg_ids)
    allowed = (seg[:, None] == seg[None, :]) & (np.arange(T)[None, :] <= np.arange(T)[:, None])
    O = np.zeros((T, H, v.shape[2]))
    for h in range(H):
        S = (q[:, h, :] @ k[:, h, :].T) * scale
        O[:, h, :] = _softmax_rows(np.where(allowed, S, -np.inf)) @ v[:, h, :]
    return O


def attention_flops(seqlens: Sequence[int], H: int, d: int) -> int:
    """Algorithmic flops of non-causal varlen attention: QK^T and PV, each
    2 * n^2 * d per head and segment."""
    return int(sum(4 * int(n) * int(n) * H * d for n in seqlens))
