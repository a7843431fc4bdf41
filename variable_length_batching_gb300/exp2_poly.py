"""Derivation of the polynomial behind the attention kernel's FMA-pipe exp2.

2^x is reduced Cody-Waite style: x = n + f with n the integer nearest to x
(found by adding 1.5 * 2^23, which rounds to an integer in the low mantissa
bits, so no floor instruction is needed) and f in [-1/2, 1/2]; then
2^x = 2^f * 2^n, and 2^n is applied by adding n to the float's exponent
field.  2^f is a cubic p(f) = c0 + c1 f + c2 f^2 + c3 f^3 chosen to minimise
the maximum relative error on [-1/2, 1/2] (a minimax fit, solved here as a
linear program on a dense grid), with p(0) = 1 pinned so that integer x map
exactly to powers of two.  Probabilities are rounded to bf16 (relative
step 2^-8) right after, so a cubic's error (about 1e-4) is far below what
that rounding keeps.

Run ``python -m variable_length_batching_gb300.exp2_poly`` to print the
coefficients and the error; the kernel's constants are these values rounded
to fp32.
"""
from __future__ import annotations

import numpy as np


def fit(degree: int = 3, grid: int = 4001, lo: float = -0.5, hi: float = 0.5):
    from scipy.optimize import linprog
    f = np.linspace(lo, hi, grid)
    target = np.exp2(f)
    # variables: c1..c_degree (c0 = 1 pinned), t
    nvar = degree + 1
    A, b = [], []
    for fi, yi in zip(f, target):
        powers = [fi ** k for k in range(1, degree + 1)]
        # |1 + sum c_k f^k - y| / y <= t  ->  two inequalities
        A.append([p / yi for p in powers] + [-1.0]); b.append(1.0 - 1.0 / yi)
        A.append([-p / yi for p in powers] + [-1.0]); b.append(-(1.0 - 1.0 / yi))
    c = np.zeros(nvar)
    c[-1] = 1.0
    res = linprog(c, A_ub=np.asarray(A), b_ub=np.asarray(b), bounds=[(None, None)] * nvar, method="highs")
    assert res.success, res.message
    coeffs = np.concatenate([[1.0], res.x[:-1]])
    return coeffs, float(res.x[-1])


def exp2_reduced(x, coeffs):
    """The device algorithm in numpy (float32): nearest-integer split via
    1.5 * 2^23, cubic on the remainder, exponent-field add."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    nf = (t - magic).astype(np.float32)
    f = (x - nf).astype(np.float32)
    c = np.asarray(coeffs, dtype=np.float32)
    p = c[3]
    for k in (2, 1, 0):
        p = (p * f + c[k]).astype(np.float32)
    n = t.view(np.int32) - np.float32(12582912.0).view(np.int32)
    return (p.view(np.int32) + (n << 23)).view(np.float32)


def evaluate(coeffs, f):
    out = np.zeros_like(f)
    for c in coeffs[::-1]:
        out = out * f + c
    return out


if __name__ == "__main__":
    coeffs, err = fit()
    c32 = coeffs.astype(np.float32)
    f = np.linspace(-0.5, 0.5, 100001)
    rel = np.abs(evaluate(c32.astype(np.float64), f) / np.exp2(f) - 1).max()
    print("coefficients (c0..c3):", [float(x) for x in c32])
    print(f"max relative error: {err:.3e} (fp32 coefficients: {rel:.3e})")
