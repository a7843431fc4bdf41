"""Planted mistakes in copies of the oracle must fail the pins.

Each case builds a wrong variant of one oracle function on the CPU (a dropped
term, a swapped index, a transposed operand, a wrong divisor) and checks that
at least one pin rejects it.  The real oracle is never modified.
"""
import numpy as np
import pytest

import _pins as pins
from oracle import partition as opart
from oracle import block as oblock
from oracle import attention as oattn


def rng(seed=0):
    return np.random.default_rng(seed)


def _fails(fn, *args):
    with pytest.raises((AssertionError, ValueError, IndexError)):
        fn(*args)


# --- partitions --------------------------------------------------------------

def inclusive_scan_partition(lengths):
    p = opart.partition(lengths)
    p.pair_off = np.concatenate([np.cumsum(p.lengths ** 2), [p.P]])
    return p


def row_major_swap_partition(lengths):
    p = opart.partition(lengths)           # row splits stride by 1 instead of N_i
    rs = []
    for i, n in enumerate(p.lengths):
        rs += [int(p.pair_off[i]) + a for a in range(int(n))]
    p.row_start = np.asarray(rs + [p.P])
    return p


def test_inclusive_scan_caught():
    _fails(pins.pin_fig2, inclusive_scan_partition)


def test_row_split_stride_caught():
    _fails(pins.pin_fig2, row_major_swap_partition)
    _fails(pins.pin_partition_bruteforce, row_major_swap_partition, [2, 3])


# --- broadcast ---------------------------------------------------------------

def broadcast_swapped_ab(lengths, s_left, s_right, W_a, W_b):
    z = oblock.pair_broadcast(lengths, s_left, s_right, W_a, W_b)
    part = opart.partition(lengths)
    out = z.copy()
    for i, n in enumerate(part.lengths):
        n = int(n)
        o = int(part.pair_off[i])
        out[o:o + n * n] = z[o:o + n * n].reshape(n, n, -1).transpose(1, 0, 2).reshape(n * n, -1)
    return out


def broadcast_transposed_weight(lengths, s_left, s_right, W_a, W_b):
    # uses W instead of W^T where shapes allow; otherwise the pad makes it fail
    Wa = W_a.T[: W_a.shape[0], : W_a.shape[1]] if W_a.shape[0] <= W_a.shape[1] else W_a
    return oblock.pair_broadcast(lengths, s_left, s_right,
                                 np.pad(Wa, ((0, W_a.shape[0] - Wa.shape[0]), (0, W_a.shape[1] - Wa.shape[1]))),
                                 W_b)


def test_broadcast_swapped_ab_caught():
    _fails(pins.pin_broadcast_onehot, broadcast_swapped_ab, rng(1))


def test_broadcast_transposed_weight_caught():
    _fails(pins.pin_broadcast_onehot, broadcast_transposed_weight, rng(1))


# --- transition --------------------------------------------------------------

def transition_no_residual(z, gamma, beta, eps, W1, b1, W2, b2):
    return oblock.pair_transition(z, gamma, beta, eps, W1, b1, W2, b2) - z


def transition_unbiased_var(z, gamma, beta, eps, W1, b1, W2, b2):
    mu = z.mean(axis=-1, keepdims=True)
    var = z.var(axis=-1, ddof=1, keepdims=True)
    ln = (z - mu) / np.sqrt(var + eps) * gamma + beta
    return z + oblock.h_theta(ln, W1, b1, W2, b2)


def transition_relu_after_second(z, gamma, beta, eps, W1, b1, W2, b2):
    ln = oblock.layer_norm(z, gamma, beta, eps)
    return z + np.maximum(oblock.linear(oblock.linear(ln, W1, b1), W2, b2), 0.0)


def transition_no_beta(z, gamma, beta, eps, W1, b1, W2, b2):
    return oblock.pair_transition(z, gamma, np.zeros_like(beta), eps, W1, b1, W2, b2)


@pytest.mark.parametrize("bad", [transition_no_residual, transition_unbiased_var,
                                 transition_relu_after_second, transition_no_beta])
def test_transition_mistakes_caught(bad):
    _fails(pins.pin_transition_library, bad, rng(4), True)


def test_dropped_residual_caught_by_identity():
    _fails(pins.pin_transition_identity, transition_no_residual, rng(5))


# --- reduce ------------------------------------------------------------------

def reduce_over_rows(lengths, z, W_g=None, b_g=None, s_in=None):
    part = opart.partition(lengths)
    zt = z.copy()
    for i, n in enumerate(part.lengths):
        n = int(n)
        o = int(part.pair_off[i])
        zt[o:o + n * n] = z[o:o + n * n].reshape(n, n, -1).transpose(1, 0, 2).reshape(n * n, -1)
    return oblock.pair_reduce(lengths, zt, W_g, b_g, s_in)


def reduce_divide_by_max(lengths, z, W_g=None, b_g=None, s_in=None):
    m, s_out = oblock.pair_reduce(lengths, z, W_g, b_g, s_in)
    part = opart.partition(lengths)
    for i, n in enumerate(part.lengths):
        m[part.cu_seqlens[i]:part.cu_seqlens[i + 1]] *= n / max(part.max_len, 1)
    return m, s_out


def reduce_no_residual(lengths, z, W_g=None, b_g=None, s_in=None):
    return oblock.pair_reduce(lengths, z, W_g, b_g, None)


def test_reduce_wrong_axis_caught():
    _fails(pins.pin_reduce_closed_form, oblock.pair_broadcast, reduce_over_rows, rng(7))


def test_reduce_wrong_divisor_caught():
    _fails(pins.pin_reduce_invariants, reduce_divide_by_max, rng(8))


def test_reduce_dropped_residual_caught():
    _fails(pins.pin_reduce_bruteforce, reduce_no_residual, rng(9))


# --- attention ---------------------------------------------------------------

def attention_no_scale(q, k, v, cu, scale=None, segments=None):
    return oattn.varlen_attention(q, k, v, cu, 1.0, segments)


def attention_no_mask(q, k, v, cu, scale=None, segments=None):
    T = q.shape[0]
    return oattn.varlen_attention(q, k, v, [0, T], scale)


def attention_off_by_one(q, k, v, cu, scale=None, segments=None):
    cu2 = [cu[0]] + [min(c + 1, cu[-1]) for c in cu[1:-1]] + [cu[-1]]
    return oattn.varlen_attention(q, k, v, cu2, scale)


def masked_leaky(q, k, v, seg, scale=None):
    return oattn.masked_full_attention(q, k, v, np.zeros(len(seg), dtype=int), scale)


def test_attention_scale_caught():
    _fails(pins.pin_attention_single_segment_sdpa, attention_no_scale, rng(13))


def test_attention_mask_caught():
    _fails(pins.pin_attention_special_cases, attention_no_mask, rng(16))
    _fails(pins.pin_attention_varlen_equals_masked, attention_no_mask, oattn.masked_full_attention, rng(15))


def test_attention_boundary_caught():
    _fails(pins.pin_attention_varlen_equals_masked, attention_off_by_one, oattn.masked_full_attention, rng(15))


def test_masked_without_mask_caught():
    _fails(pins.pin_attention_masked_core_math, masked_leaky, rng(14))


def _segment_attention_mask(allow_fn):
    """A copy of the per-segment attention with a different causal mask."""
    def seg_attn(q, k, v, scale, causal=False):
        nq, H, _ = q.shape
        nk = k.shape[0]
        allowed = allow_fn(nq, nk) if causal else np.ones((nq, nk), dtype=bool)
        O = np.zeros((nq, H, v.shape[2]))
        lse = np.full((H, nq), -np.inf)
        for h in range(H):
            S = (q[:, h, :] @ k[:, h, :].T) * scale
            for i in range(nq):
                if allowed[i].any():
                    s = S[i, allowed[i]]
                    e = np.exp(s - s.max())
                    O[i, h, :] = (e / e.sum()) @ v[allowed[i], h, :]
                    lse[h, i] = s.max() + np.log(e.sum())
        return O, lse
    return seg_attn


def _with_segment(seg_attn):
    def attn(q, k, v, cu, scale=None, segments=None, causal=False, cu_seqlens_k=None):
        orig = oattn.segment_attention
        oattn.segment_attention = seg_attn
        try:
            return oattn.varlen_attention(q, k, v, cu, scale, segments, causal, cu_seqlens_k)
        finally:
            oattn.segment_attention = orig
    return attn


strict_causal = _with_segment(_segment_attention_mask(
    lambda nq, nk: np.arange(nk)[None, :] < np.arange(nq)[:, None] + (nk - nq)))
top_left_causal = _with_segment(_segment_attention_mask(
    lambda nq, nk: np.arange(nk)[None, :] <= np.arange(nq)[:, None]))


def test_causal_strict_mask_caught():
    _fails(pins.pin_attention_causal_sdpa, strict_causal, rng(17))
    _fails(pins.pin_attention_causal_masked, strict_causal, oattn.masked_full_attention_causal, rng(19))


def test_causal_top_left_alignment_caught():
    _fails(pins.pin_attention_cross_sdpa, top_left_causal, rng(18))


def test_cross_uses_query_offsets_for_keys_caught():
    def same_cu(q, k, v, cu, scale=None, segments=None, causal=False, cu_seqlens_k=None):
        T = q.shape[0]
        return oattn.varlen_attention(q, k[:T] if k.shape[0] >= T else np.resize(k, q.shape),
                                      v[:T] if v.shape[0] >= T else np.resize(v, q.shape),
                                      cu, scale, segments, causal, None)
    _fails(pins.pin_attention_cross_sdpa, same_cu, rng(18))


# --- rectangular pairs ---------------------------------------------------------

def rect_partition_row_stride_n(rows, cols):
    p = opart.partition_rect(rows, cols)      # rows stride by N_i instead of M_i
    rs = []
    for i, n in enumerate(p.rows):
        rs += [int(p.pair_off[i]) + a * int(n) for a in range(int(n))]
    p.row_start = np.asarray(rs + [p.P])
    return p


def rect_reduce_divides_by_rows(rows, cols, z, W_g=None, b_g=None, s_in=None):
    m, s_out = oblock.pair_reduce_rect(rows, cols, z, W_g, b_g, s_in)
    p = opart.partition_rect(rows, cols)
    for i in range(len(p.rows)):
        n, mm = int(p.rows[i]), int(p.cols[i])
        if n and mm:
            m[p.cu_rows[i]:p.cu_rows[i + 1]] *= mm / n
    return m, s_out


def rect_broadcast_cols_from_row_offsets(rows, cols, s_row, s_col, W_a, W_b):
    p = opart.partition_rect(rows, cols)
    z = np.zeros((p.P, W_a.shape[0]))
    for i in range(len(p.rows)):
        n, m = int(p.rows[i]), int(p.cols[i])
        U = oblock.linear(s_row[p.cu_rows[i]:p.cu_rows[i + 1]], W_a)
        V = oblock.linear(np.resize(s_col[p.cu_rows[i]:], (max(m, 1), s_col.shape[1]))[:m], W_b)
        for a in range(n):
            for b in range(m):
                z[int(p.pair_off[i]) + a * m + b] = U[a] + V[b]
    return z


def test_rect_row_stride_caught():
    _fails(pins.pin_rect_partition_bruteforce, rect_partition_row_stride_n, [2, 3], [4, 1])


def test_rect_divisor_caught():
    _fails(pins.pin_rect_reduce_closed_form, oblock.pair_broadcast_rect, rect_reduce_divides_by_rows, rng(23))


def test_rect_column_offsets_caught():
    _fails(pins.pin_rect_broadcast_onehot, rect_broadcast_cols_from_row_offsets, rng(21))


# --- SwiGLU transition ----------------------------------------------------------

def swiglu_swapped(P, gamma, beta, eps, W1, b1, W3, b3, W2, b2):
    return oblock.transition_swiglu(P, gamma, beta, eps, W3, b3, W1, b1, W2, b2)   # value gated


def swiglu_sigmoid(P, gamma, beta, eps, W1, b1, W3, b3, W2, b2):
    y = oblock.layer_norm(P, gamma, beta, eps)
    g = oblock.linear(y, W1, b1)
    return P + oblock.linear(g / g * (1 / (1 + np.exp(-g))) * oblock.linear(y, W3, b3), W2, b2)


def swiglu_no_residual(P, gamma, beta, eps, W1, b1, W3, b3, W2, b2):
    return oblock.transition_swiglu(P, gamma, beta, eps, W1, b1, W3, b3, W2, b2) - P


def test_swiglu_mistakes_caught():
    _fails(pins.pin_swiglu_library, swiglu_swapped, rng(25))
    _fails(pins.pin_swiglu_library, swiglu_sigmoid, rng(25))
    _fails(pins.pin_swiglu_library, swiglu_no_residual, rng(25))
    _fails(pins.pin_swiglu_zero_gate, swiglu_no_residual, rng(27))


def test_silu_mistake_caught():
    _fails(pins.pin_silu, lambda x: 1 / (1 + np.exp(-x)))


# --- attention backward -----------------------------------------------------------

def backward_without_rowsum(q, k, v, do, cu, scale=None, causal=False, cu_seqlens_k=None, segments=None):
    """dS = P * dP (the rowsum(dO * O) term dropped)."""
    orig = oattn.segment_attention_backward

    def seg(q, k, v, do, scale, causal=False):
        nq, H, d = q.shape
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for h in range(H):
            S = (q[:, h, :] @ k[:, h, :].T) * scale
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            dP = do[:, h, :] @ v[:, h, :].T
            dS = P * dP
            dv[:, h, :] = P.T @ do[:, h, :]
            dq[:, h, :] = scale * dS @ k[:, h, :]
            dk[:, h, :] = scale * dS.T @ q[:, h, :]
        return dq, dk, dv
    oattn.segment_attention_backward = seg
    try:
        return oattn.varlen_attention_backward(q, k, v, do, cu, scale, causal, cu_seqlens_k, segments)
    finally:
        oattn.segment_attention_backward = orig


def test_backward_rowsum_caught():
    _fails(pins.pin_attention_backward_autograd, backward_without_rowsum, rng(28))


# --- Eq. 5 loss and the block's gradients ------------------------------------

def _mutated_backward(old, new):
    """A copy of oracle.block_backward with one planted mistake (source
    replacement), loaded as a separate module; the real one is untouched."""
    import importlib.util
    import os
    import oracle
    path = os.path.join(os.path.dirname(oracle.__file__), "block_backward.py")
    src = open(path).read()
    assert src.count(old) == 1, old
    spec = importlib.util.spec_from_loader("oracle._mutated_block_backward", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(src.replace(old, new), path, "exec"), mod.__dict__)
    return mod


BACKWARD_MISTAKES = [
    # the column mean's 1/N dropped in the reduce backward
    ("dPt = dP_tilde + dM[:, None, :] / N", "dPt = dP_tilde + dM[:, None, :]"),
    # ReLU's mask forgotten
    ("dA = dH * (A > 0)", "dA = dH"),
    # the LayerNorm backward without its xhat term
    ("- xhat * (dxhat * xhat).mean(axis=-1, keepdims=True)) / sigma", ") / sigma"),
    # column and row sums of the broadcast swapped
    ("dU = dP.sum(axis=1)", "dU = dP.sum(axis=0)"),
    # the singles' residual path dropped
    ("dX = dX_tilde.copy()", "dX = 0 * dX_tilde"),
    # Eq. 5's weights swapped between the two terms
    ("return 1.0 + i / B, 1.5 - i / (2.0 * B)", "return 1.5 - i / (2.0 * B), 1.0 + i / B"),
    # pair term normalised by sum N_i instead of sum N_i^2
    ("dz[c0:c1] = 2.0 * beta[i] * z_tilde[c0:c1] / (C_p * part.P)",
     "dz[c0:c1] = 2.0 * beta[i] * z_tilde[c0:c1] / (C_p * part.T)"),
]


@pytest.mark.parametrize("old,new", BACKWARD_MISTAKES)
def test_backward_mistakes_caught(old, new):
    mod = _mutated_backward(old, new)
    _fails(pins.pin_block_backward_autograd, mod.block_loss_and_grads, oblock.block_packed, rng(5))


def test_eq5_weight_mistake_caught_by_hand_values():
    mod = _mutated_backward(*BACKWARD_MISTAKES[5])
    _fails(pins.pin_eq5_weights, mod.eq5_sample_weights)
