"""Oracle for the sample-weighted loss of the single->pair->single block and
for the block's gradients.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "DanLing NestedTensor: Composable Multi-Ragged Tensors for Deep
Learning":

* Appendix A.1, Eq. 5: both outputs of Eq. 1 feed an eager, sample-weighted
  squared loss,

      L = sum_i alpha_i ||X~_i||_F^2 / (S C sum_i N_i)
        + sum_i beta_i  ||P~_i||_F^2 / (S C_p sum_i N_i M_i),

  with alpha_i = 1 + i / B, beta_i = 1.5 - i / (2 B) for i = 0 .. B-1,
  S = 1 for leading layouts (the packed layout here), M_i = N_i for square
  pairs; the squared sums accumulate in at least fp32 (here fp64).
* Section 4.1 "Protocol" and Appendix A.1: the measured step covers the
  forward computation, this loss and the backward; section 3.4: gradients
  flow from the eager loss back through the pair update, the reduction and
  the projections of Eq. 1.

The gradients are the chain rule of Eq. 1 (see ``block.block_sample``),
written out per sample, densely, in the order the forward runs backwards:

    dX~ = dL/dX~,  dP~ = dL/dP~ (given)
    X~  = X + M W_g^T + b_g:   dM = dX~ W_g,  dW_g = dX~^T M,  db_g = sum dX~
    M[a] = (1/N) sum_b P~[a, b]:   dP~[a, b] += dM[a] / N
    P~  = P + h(Y) W2^T + b2,  h = ReLU(A),  A = Y W1^T + b1,  Y = LN(P):
        dH = dP~ W2,  dW2 = dP~^T H,  db2 = sum dP~
        dA = dH * [A > 0],  dW1 = dA^T Y,  db1 = sum dA,  dY = dA W1
        LN with xhat = (P - mu) / sigma, sigma = sqrt(var + eps):
          dgamma = sum dY * xhat,  dbeta = sum dY,  dxhat = dY * gamma,
          dP_ln = (dxhat - mean(dxhat) - xhat * mean(dxhat * xhat)) / sigma
        dP = dP~ + dP_ln
    P[a, b] = U[a] + V[b],  U = X W_a^T,  V = X W_b^T:
        dU[a] = sum_b dP[a, b],  dV[b] = sum_a dP[a, b]
        dW_a = dU^T X,  dW_b = dV^T X,  dX += dU W_a + dV W_b

(the means in the LayerNorm backward run over the C_p features of one cell;
ReLU's derivative is taken as 1 where A > 0 and 0 elsewhere).  Weight
gradients are sums over every sample's cells and rows.  Everything is
float64; inputs are the exact values handed to the GPU.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Sequence

import numpy as np

from .block import Weights, linear
from .partition import partition


def eq5_sample_weights(B: int):
    """alpha_i = 1 + i / B and beta_i = 1.5 - i / (2 B), i = 0 .. B-1 (Eq. 5)."""
    i = np.arange(B, dtype=np.float64)
    return 1.0 + i / B, 1.5 - i / (2.0 * B)


def eq5_loss(lengths: Sequence[int], s_out: np.ndarray, z_tilde: np.ndarray) -> float:
    """Eq. 5 on the packed outputs of one block (square pairs, S = 1):
    per-sample squared Frobenius norms of X~_i (rows of s_out) and P~_i
    (cells of z_tilde), weighted and normalised as the equation states."""
    part = partition(lengths)
    B = len(part.lengths)
    alpha, beta = eq5_sample_weights(B)
    C, C_p = s_out.shape[1], z_tilde.shape[1]
    T, P = part.T, part.P
    lx = lp = 0.0
    for i in range(B):
        X = s_out[part.cu_seqlens[i]:part.cu_seqlens[i + 1]]
        Pt = z_tilde[part.pair_off[i]:part.pair_off[i + 1]]
        lx += alpha[i] * float((X * X).sum())
        lp += beta[i] * float((Pt * Pt).sum())
    return (lx / (C * T) if T else 0.0) + (lp / (C_p * P) if P else 0.0)


def eq5_loss_grads(lengths: Sequence[int], s_out: np.ndarray, z_tilde: np.ndarray):
    """dL/ds_out and dL/dz_tilde of Eq. 5: 2 alpha_i X~_i / (C sum N_i) and
    2 beta_i P~_i / (C_p sum N_i^2), row by row and cell by cell."""
    part = partition(lengths)
    B = len(part.lengths)
    alpha, beta = eq5_sample_weights(B)
    C, C_p = s_out.shape[1], z_tilde.shape[1]
    ds = np.zeros_like(s_out)
    dz = np.zeros_like(z_tilde)
    for i in range(B):
        r0, r1 = part.cu_seqlens[i], part.cu_seqlens[i + 1]
        c0, c1 = part.pair_off[i], part.pair_off[i + 1]
        ds[r0:r1] = 2.0 * alpha[i] * s_out[r0:r1] / (C * part.T)
        dz[c0:c1] = 2.0 * beta[i] * z_tilde[c0:c1] / (C_p * part.P)
    return ds, dz


@dataclass
class BlockGrads:
    ds: np.ndarray        # (T, C) gradient of the singles
    dW_a: np.ndarray      # (C_p, C)
    dW_b: np.ndarray      # (C_p, C)
    dgamma: np.ndarray    # (C_p,)
    dbeta: np.ndarray     # (C_p,)
    dW1: np.ndarray       # (H_t, C_p)
    db1: np.ndarray       # (H_t,)
    dW2: np.ndarray       # (C_p, H_t)
    db2: np.ndarray       # (C_p,)
    dW_g: np.ndarray      # (C, C_p)
    db_g: np.ndarray      # (C,)


def block_backward_sample(X: np.ndarray, w: Weights, dX_tilde: np.ndarray, dP_tilde: np.ndarray):
    """Gradients of one sample's block (square pairs) for upstream gradients
    dX~ (N, C) and dP~ (N, N, C_p): returns (dX, dict of weight gradients)."""
    N = X.shape[0]
    # forward, keeping what the backward needs
    U = linear(X, w.W_a)
    V = linear(X, w.W_b)
    P = U[:, None, :] + V[None, :, :]                          # (N, N, C_p)
    mu = P.mean(axis=-1, keepdims=True)
    sigma = np.sqrt(((P - mu) ** 2).mean(axis=-1, keepdims=True) + w.eps)
    xhat = (P - mu) / sigma
    Y = xhat * w.gamma + w.beta                                # = layer_norm(P, ...)
    A = linear(Y, w.W1, w.b1)                                  # (N, N, H_t)
    H = np.maximum(A, 0.0)
    P_tilde = P + linear(H, w.W2, w.b2)
    M = P_tilde.sum(axis=1) / N                                # (N, C_p)
    # X~ = X + M W_g^T + b_g
    dX = dX_tilde.copy()
    dM = dX_tilde @ w.W_g                                      # (N, C_p)
    g = {"dW_g": dX_tilde.T @ M, "db_g": dX_tilde.sum(axis=0)}
    # M[a] = (1/N) sum_b P~[a, b]
    dPt = dP_tilde + dM[:, None, :] / N
    # P~ = P + H W2^T + b2
    dH = dPt @ w.W2                                            # (N, N, H_t)
    g["dW2"] = np.einsum("abc,abh->ch", dPt, H, optimize=True)
    g["db2"] = dPt.sum(axis=(0, 1))
    dA = dH * (A > 0)
    g["dW1"] = np.einsum("abh,abc->hc", dA, Y, optimize=True)
    g["db1"] = dA.sum(axis=(0, 1))
    dY = dA @ w.W1                                             # (N, N, C_p)
    g["dgamma"] = (dY * xhat).sum(axis=(0, 1))
    g["dbeta"] = dY.sum(axis=(0, 1))
    dxhat = dY * w.gamma
    dP_ln = (dxhat - dxhat.mean(axis=-1, keepdims=True)
             - xhat * (dxhat * xhat).mean(axis=-1, keepdims=True)) / sigma
    dP = dPt + dP_ln
    # P[a, b] = U[a] + V[b]
    dU = dP.sum(axis=1)                                        # (N, C_p)
    dV = dP.sum(axis=0)
    g["dW_a"] = dU.T @ X
    g["dW_b"] = dV.T @ X
    dX = dX + dU @ w.W_a + dV @ w.W_b
    return dX, g


def block_backward_packed(lengths: Sequence[int], s: np.ndarray, w: Weights, ds_out: np.ndarray,
                          dz_tilde: np.ndarray) -> BlockGrads:
    """``block_backward_sample`` on every sample (upstream gradients in the
    packed layout of Eq. 2/3), with the weight gradients summed over the
    batch."""
    part = partition(lengths)
    C, C_p, H_t = s.shape[1], w.W_a.shape[0], w.W1.shape[0]
    ds = np.zeros_like(s)
    acc = {"dW_a": np.zeros((C_p, C)), "dW_b": np.zeros((C_p, C)), "dgamma": np.zeros(C_p),
           "dbeta": np.zeros(C_p), "dW1": np.zeros((H_t, C_p)), "db1": np.zeros(H_t),
           "dW2": np.zeros((C_p, H_t)), "db2": np.zeros(C_p), "dW_g": np.zeros((C, C_p)), "db_g": np.zeros(C)}
    for i, N in enumerate(part.lengths):
        N = int(N)
        if N == 0:
            continue
        r0, r1 = part.cu_seqlens[i], part.cu_seqlens[i + 1]
        o = int(part.pair_off[i])
        dX, g = block_backward_sample(s[r0:r1], w, ds_out[r0:r1], dz_tilde[o:o + N * N].reshape(N, N, C_p))
        ds[r0:r1] = dX
        for k, v in g.items():
            acc[k] += v
    return BlockGrads(ds=ds, **acc)


def block_loss_and_grads(lengths: Sequence[int], s: np.ndarray, w: Weights, z_tilde: np.ndarray,
                         s_out: np.ndarray):
    """Eq. 5 on the block's outputs and the gradients of that loss with
    respect to the singles and every parameter (one training step's
    backward for a lone block)."""
    ds_out, dz = eq5_loss_grads(lengths, s_out, z_tilde)
    return eq5_loss(lengths, s_out, z_tilde), block_backward_packed(lengths, s, w, ds_out, dz)
