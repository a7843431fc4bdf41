"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each pin takes the oracle callables it checks as arguments, so the same pin
runs against the real oracle (``test_oracle_pins.py``) and against copies
with a planted mistake (``test_oracle_mutations.py``), which must fail it.
None of these checks re-types the oracle's own formula: each compares it
with a printed value, a closed form, a library routine on a special case,
an invariant or a brute-force enumeration.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

from _helpers import golden


# ----------------------------------------------------------------------------
# Partitions ("DanLing NestedTensor" Eq. 2, Eq. 3, Figure 2, Appendix A)
# ----------------------------------------------------------------------------

def pin_fig2(partition):
    g = golden("fig2_partition.json")
    p = partition(g["lengths"])
    pr, dv = g["printed"], g["derived_from_prose"]
    assert p.T == pr["single_positions"]
    assert p.P == pr["pair_cells"]
    assert list(p.cu_seqlens) == pr["single_offsets"]
    assert list(p.pair_off) == pr["pair_offsets"]
    assert len(p.row_start) == pr["second_level_split_entries"]
    assert list(p.row_start) == dv["second_level_splits"]


def pin_partition_invariants(partition, lengths):
    p = partition(lengths)
    N = np.asarray(lengths, dtype=np.int64)
    # Appendix A: o_0 = 0, o_{i+1} - o_i = p_i, o_B = T
    assert p.cu_seqlens[0] == 0 and p.pair_off[0] == 0
    assert np.array_equal(np.diff(p.cu_seqlens), N)
    assert np.array_equal(np.diff(p.pair_off), N * N)
    assert p.cu_seqlens[-1] == p.T == N.sum()
    assert p.pair_off[-1] == p.P == (N * N).sum()
    assert len(p.row_start) == 1 + N.sum()
    assert p.max_len == (N.max() if len(N) else 0)


def pin_partition_bruteforce(partition, lengths):
    """Walk every (sample, a, b) in order: Eq. 3 must number the cells
    0, 1, 2, ... consecutively, and each row's first cell is its split."""
    p = partition(lengths)
    cell = 0
    row = 0
    for i, n in enumerate(lengths):
        for a in range(n):
            assert p.row_start[row] == cell
            assert p.row_sample[row] == i
            for b in range(n):
                assert p.pair_off[i] + a * n + b == cell
                cell += 1
            row += 1
    assert row == p.T and cell == p.P and p.row_start[-1] == cell


# ----------------------------------------------------------------------------
# Block ("DanLing NestedTensor" Eq. 1, Eq. 4)
# ----------------------------------------------------------------------------

def pin_broadcast_onehot(pair_broadcast, rng):
    """One-hot projections select single features: with W_a picking feature
    f of X[a] and W_b zero, cell (a, b) holds X[a, f]; swapped, it holds
    X[b, g].  Fixes the order of a and b and the orientation of W."""
    lengths = [3, 1, 4, 0, 2]
    C, C_p = 5, 3
    T = sum(lengths)
    s = rng.standard_normal((T, C))
    Wsel = np.zeros((C_p, C))
    Wsel[0, 2] = 1.0
    Wsel[1, 4] = 1.0
    Wsel[2, 0] = 1.0
    Z = np.zeros((C_p, C))
    za = pair_broadcast(lengths, s, s, Wsel, Z)
    zb = pair_broadcast(lengths, s, s, Z, Wsel)
    z0 = pair_broadcast(lengths, s, s, Z, Z)
    assert za.shape == (sum(n * n for n in lengths), C_p)
    assert np.all(z0 == 0.0)
    cell, start = 0, 0
    for n in lengths:
        for a in range(n):
            for b in range(n):
                assert np.array_equal(za[cell], s[start + a, [2, 4, 0]])
                assert np.array_equal(zb[cell], s[start + b, [2, 4, 0]])
                cell += 1
        start += n


def pin_broadcast_left_right(pair_broadcast, rng):
    """Distinct left/right singles: cell (a, b) = X_L[a] W_a^T + X_R[b] W_b^T,
    checked with torch's linear on each cell (brute force)."""
    lengths = [2, 3]
    C, C_p = 4, 3
    T = sum(lengths)
    sL, sR = rng.standard_normal((T, C)), rng.standard_normal((T, C))
    Wa, Wb = rng.standard_normal((C_p, C)), rng.standard_normal((C_p, C))
    z = pair_broadcast(lengths, sL, sR, Wa, Wb)
    tL, tR = torch.from_numpy(sL), torch.from_numpy(sR)
    ta, tb = torch.from_numpy(Wa), torch.from_numpy(Wb)
    cell, start = 0, 0
    for n in lengths:
        for a in range(n):
            for b in range(n):
                ref = F.linear(tL[start + a], ta) + F.linear(tR[start + b], tb)
                assert np.allclose(z[cell], ref.numpy(), rtol=1e-13, atol=1e-13)
                cell += 1
        start += n


def pin_transition_library(pair_transition, rng, biases=True):
    """On any cells, LN -> Linear -> ReLU -> Linear plus residual equals
    torch.nn.functional's layer_norm / linear / relu in float64."""
    P, C_p, H = 37, 8, 24
    z = rng.standard_normal((P, C_p)) * 3.0 + 0.5
    gamma = 1.0 + 0.1 * rng.standard_normal(C_p)
    beta = 0.1 * rng.standard_normal(C_p)
    W1, W2 = rng.standard_normal((H, C_p)), rng.standard_normal((C_p, H))
    b1 = rng.standard_normal(H) if biases else None
    b2 = rng.standard_normal(C_p) if biases else None
    got = pair_transition(z, gamma, beta, 1e-5, W1, b1, W2, b2)
    tz = torch.from_numpy(z)
    ln = F.layer_norm(tz, (C_p,), torch.from_numpy(gamma), torch.from_numpy(beta), 1e-5)
    hid = F.relu(F.linear(ln, torch.from_numpy(W1), None if b1 is None else torch.from_numpy(b1)))
    ref = tz + F.linear(hid, torch.from_numpy(W2), None if b2 is None else torch.from_numpy(b2))
    assert np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def pin_transition_identity(pair_transition, rng):
    """W2 = 0 and b2 = 0: the update vanishes and z~ = z exactly."""
    z = rng.standard_normal((11, 6))
    out = pair_transition(z, np.ones(6), np.zeros(6), 1e-5, rng.standard_normal((10, 6)),
                          rng.standard_normal(10), np.zeros((6, 10)), None)
    assert np.array_equal(out, z)


def pin_layernorm_constant(layer_norm, rng):
    """A constant-feature cell normalises to beta exactly."""
    beta = rng.standard_normal(7)
    x = np.full((3, 7), 2.5)
    assert np.array_equal(layer_norm(x, rng.standard_normal(7), beta, 1e-5), np.broadcast_to(beta, (3, 7)))


def pin_reduce_closed_form(pair_broadcast, pair_reduce, rng):
    """Without a transition, mean_b (U[a] + V[b]) = U[a] + mean_b V[b]."""
    lengths = [4, 1, 0, 3, 6]
    C, C_p = 5, 4
    T = sum(lengths)
    s = rng.standard_normal((T, C))
    Wa, Wb = rng.standard_normal((C_p, C)), rng.standard_normal((C_p, C))
    z = pair_broadcast(lengths, s, s, Wa, Wb)
    m, _ = pair_reduce(lengths, z)
    U, V = s @ Wa.T, s @ Wb.T
    start = 0
    for n in lengths:
        for a in range(n):
            ref = U[start + a] + V[start:start + n].sum(axis=0) / n
            assert np.allclose(m[start + a], ref, rtol=1e-12, atol=1e-12)
        start += n


def pin_reduce_invariants(pair_reduce, rng):
    """A per-sample constant pair state reduces to that constant; N_i = 1
    returns the cell itself; sum_a N_i m[a] equals the sample's cell sum."""
    lengths = [3, 1, 5]
    C_p = 4
    consts = rng.standard_normal((3, C_p))
    z = np.concatenate([np.broadcast_to(consts[i], (n * n, C_p)) for i, n in enumerate(lengths)])
    m, _ = pair_reduce(lengths, z)
    assert np.allclose(m[:3], consts[0], rtol=1e-14, atol=1e-14)
    assert np.array_equal(m[3], consts[1])
    assert np.allclose(m[4:], consts[2], rtol=1e-14, atol=1e-14)
    z = rng.standard_normal((sum(n * n for n in lengths), C_p))
    m, _ = pair_reduce(lengths, z)
    assert np.array_equal(m[3], z[9])
    cell, row = 0, 0
    for n in lengths:
        assert np.allclose(n * m[row:row + n].sum(axis=0), z[cell:cell + n * n].sum(axis=0),
                           rtol=1e-12, atol=1e-12)
        cell += n * n
        row += n


def pin_reduce_bruteforce(pair_reduce, rng):
    """Eq. 4 walked cell by cell: rows of sample i start at eta_i, cells at
    o_i + a N_i + b; the g projection and residual via torch."""
    lengths = [2, 3, 1]
    C_p, C = 3, 4
    z = rng.standard_normal((sum(n * n for n in lengths), C_p))
    s_in = rng.standard_normal((sum(lengths), C))
    Wg, bg = rng.standard_normal((C, C_p)), rng.standard_normal(C)
    m, s_out = pair_reduce(lengths, z, Wg, bg, s_in)
    o, eta = 0, 0
    for n in lengths:
        for a in range(n):
            acc = np.zeros(C_p)
            for b in range(n):
                acc = acc + z[o + a * n + b]
            assert np.allclose(m[eta + a], acc / n, rtol=1e-13, atol=1e-13)
            ref = torch.from_numpy(s_in[eta + a]) + F.linear(torch.from_numpy(acc / n),
                                                             torch.from_numpy(Wg), torch.from_numpy(bg))
            assert np.allclose(s_out[eta + a], ref.numpy(), rtol=1e-12, atol=1e-12)
        o += n * n
        eta += n


def pin_packed_equals_padded(block_packed, block_padded_gathered, weights, lengths, s):
    """Packed results equal the padded-then-gathered ones on valid cells
    ("DanLing NestedTensor" Appendix A, reference semantics)."""
    a = block_packed(lengths, s, weights)
    b = block_padded_gathered(lengths, s, weights)
    for name in ("z", "z_tilde", "m", "s_out"):
        x, y = getattr(a, name), getattr(b, name)
        assert x.shape == y.shape, name
        assert np.allclose(x, y, rtol=1e-11, atol=1e-11), name


# ----------------------------------------------------------------------------
# Attention ("Variable-length attention and data packing")
# ----------------------------------------------------------------------------

def pin_attention_single_segment_sdpa(varlen_attention, rng):
    """One segment is plain dense attention: torch's scaled_dot_product_attention
    (float64, non-causal, default scale d^-1/2)."""
    n, H, d = 13, 3, 8
    q, k, v = (rng.standard_normal((n, H, d)) for _ in range(3))
    O, lse = varlen_attention(q, k, v, [0, n])
    tq, tk, tv = (torch.from_numpy(x).permute(1, 0, 2) for x in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv).permute(1, 0, 2).numpy()
    assert np.allclose(O, ref, rtol=1e-12, atol=1e-12)
    S = torch.einsum("hnd,hmd->hnm", tq, tk) / np.sqrt(d)
    assert np.allclose(lse, torch.logsumexp(S, dim=-1).numpy(), rtol=1e-12, atol=1e-12)


def pin_attention_masked_core_math(masked_full_attention, rng):
    """The page's nine-token example: masked rows sum to one with zero
    cross-sample mass; without the mask the softmax leaks above 1e-3."""
    g = golden("core_math_mask.json")
    seg = np.asarray(g["segment_ids"])
    T, H, d = len(seg), 2, 4
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    _, A = masked_full_attention(q, k, v, seg)
    block = seg[:, None] == seg[None, :]
    assert np.all(A[:, ~block] == 0.0)
    assert np.allclose(A.sum(axis=-1), 1.0, rtol=0, atol=1e-14)
    _, A_leak = masked_full_attention(q, k, v, np.zeros(T, dtype=int))
    assert A_leak[:, ~block].max() > g["leak_threshold"]


def pin_attention_varlen_equals_masked(varlen_attention, masked_full_attention, rng):
    """Per-segment attention equals the full T x T block-diagonal masked
    attention on a tiny stream (brute force)."""
    g = golden("core_math_mask.json")
    cu = g["cu_seqlens"] + [12]   # add a fourth segment of 3 tokens
    seg = np.repeat(np.arange(len(cu) - 1), np.diff(cu))
    T, H, d = cu[-1], 2, 5
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    O1, _ = varlen_attention(q, k, v, cu)
    O2, _ = masked_full_attention(q, k, v, seg)
    assert np.allclose(O1, O2, rtol=1e-12, atol=1e-12)


def pin_attention_special_cases(varlen_attention, rng):
    """A length-1 segment returns its own v; a segment whose v is constant
    returns that constant; changing one segment's tokens leaves every other
    segment's output bit-identical (zero leakage)."""
    cu = [0, 1, 5, 5, 12]
    T, H, d = 12, 2, 4
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    v[5:12] = rng.standard_normal((1, H, d))
    O, _ = varlen_attention(q, k, v, cu)
    assert np.allclose(O[0], v[0], rtol=1e-15, atol=1e-15)
    assert np.allclose(O[5:12], v[5:12], rtol=1e-13, atol=1e-13)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[1:5] += 1.0
    k2[1:5] *= -2.0
    v2[1:5] = rng.standard_normal((4, H, d))
    O2, _ = varlen_attention(q2, k2, v2, cu)
    assert np.array_equal(O2[:1], O[:1]) and np.array_equal(O2[5:], O[5:])
    assert not np.allclose(O2[1:5], O[1:5])


def pin_attention_causal_sdpa(varlen_attention, rng):
    """Causal self-attention of one segment is torch's SDPA with is_causal."""
    n, H, d = 11, 2, 8
    q, k, v = (rng.standard_normal((n, H, d)) for _ in range(3))
    O, _ = varlen_attention(q, k, v, [0, n], causal=True)
    tq, tk, tv = (torch.from_numpy(x).permute(1, 0, 2) for x in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True).permute(1, 0, 2).numpy()
    assert np.allclose(O, ref, rtol=1e-12, atol=1e-12)


def pin_attention_cross_sdpa(varlen_attention, rng):
    """Cross-attention, query and key lengths differ: each segment is SDPA of
    its queries against its own keys (non-causal), and with the causal flag the
    mask is torch.ones(n_q, n_k).tril(n_k - n_q) (bottom-right alignment)."""
    cu_q, cu_k = [0, 3, 9, 9, 13], [0, 7, 10, 12, 20]
    H, d = 2, 5
    q = rng.standard_normal((cu_q[-1], H, d))
    k, v = (rng.standard_normal((cu_k[-1], H, d)) for _ in range(2))
    for causal in (False, True):
        O, lse = varlen_attention(q, k, v, cu_q, causal=causal, cu_seqlens_k=cu_k)
        for b in range(len(cu_q) - 1):
            ql, qh, kl, kh = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
            if qh == ql:
                continue
            tq = torch.from_numpy(q[ql:qh]).permute(1, 0, 2)
            tk = torch.from_numpy(k[kl:kh]).permute(1, 0, 2)
            tv = torch.from_numpy(v[kl:kh]).permute(1, 0, 2)
            mask = None
            if causal:
                mask = torch.ones(qh - ql, kh - kl, dtype=torch.bool).tril(kh - kl - (qh - ql))
            ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask).permute(1, 0, 2).numpy()
            assert np.allclose(O[ql:qh], ref, rtol=1e-12, atol=1e-12)


def pin_attention_causal_masked(varlen_attention, masked_full_attention_causal, rng):
    """Per-segment causal attention equals the full T x T masked form."""
    cu = [0, 4, 5, 12]
    seg = np.repeat(np.arange(3), np.diff(cu))
    q, k, v = (rng.standard_normal((12, 2, 4)) for _ in range(3))
    O1, _ = varlen_attention(q, k, v, cu, causal=True)
    assert np.allclose(O1, masked_full_attention_causal(q, k, v, seg), rtol=1e-12, atol=1e-12)
    # the first query of every segment sees only its own key: O = v
    for b in range(3):
        assert np.allclose(O1[cu[b]], v[cu[b]], rtol=1e-14, atol=1e-14)


# ----------------------------------------------------------------------------
# Rectangular pairs ("DanLing NestedTensor" section 3.2 "Consuming one logical
# axis", Eq. 4; Appendix A.1, rectangular variant)
# ----------------------------------------------------------------------------

def pin_rect_partition_bruteforce(partition_rect, rows, cols):
    """Walking every (sample, a, b) with b < M_i in order numbers the cells
    0, 1, 2, ...; each row starts at its split; rows and columns scan
    separately; M = N gives the square partition."""
    p = partition_rect(rows, cols)
    cell, row = 0, 0
    for i, (n, m) in enumerate(zip(rows, cols)):
        assert p.cu_rows[i] == sum(rows[:i]) and p.cu_cols[i] == sum(cols[:i])
        for a in range(n):
            assert p.row_start[row] == cell and p.row_sample[row] == i
            cell += m
            row += 1
    assert row == p.T_rows == sum(rows) and cell == p.P == sum(n * m for n, m in zip(rows, cols))
    assert p.T_cols == sum(cols) and p.row_start[-1] == p.P
    assert np.array_equal(np.diff(p.pair_off), np.asarray(rows) * np.asarray(cols))


def pin_rect_square_case(partition_rect, partition, lengths):
    """A rectangular partition with M_i = N_i is the square partition."""
    r, s = partition_rect(lengths, lengths), partition(lengths)
    assert np.array_equal(r.pair_off, s.pair_off) and np.array_equal(r.row_start, s.row_start)
    assert np.array_equal(r.cu_rows, s.cu_seqlens) and np.array_equal(r.cu_cols, s.cu_seqlens)


def pin_rect_broadcast_onehot(pair_broadcast_rect, rng):
    """One-hot projections: with W_b = 0 cell (a, b) holds the selected
    features of row single a; with W_a = 0, those of column single b.  Rows
    and columns come from their own inputs at their own offsets."""
    rows, cols = [2, 0, 3, 1], [3, 2, 1, 0]
    C, C_p = 4, 2
    s_row = rng.standard_normal((sum(rows), C))
    s_col = rng.standard_normal((sum(cols), C))
    Wsel = np.zeros((C_p, C))
    Wsel[0, 3] = 1.0
    Wsel[1, 1] = 1.0
    Z = np.zeros((C_p, C))
    za = pair_broadcast_rect(rows, cols, s_row, s_col, Wsel, Z)
    zb = pair_broadcast_rect(rows, cols, s_row, s_col, Z, Wsel)
    assert za.shape == (sum(n * m for n, m in zip(rows, cols)), C_p)
    cell, r0, c0 = 0, 0, 0
    for n, m in zip(rows, cols):
        for a in range(n):
            for b in range(m):
                assert np.array_equal(za[cell], s_row[r0 + a, [3, 1]])
                assert np.array_equal(zb[cell], s_col[c0 + b, [3, 1]])
                cell += 1
        r0 += n
        c0 += m


def pin_rect_broadcast_library(pair_broadcast_rect, rng):
    """Every cell equals torch's linear of its row single plus its column single."""
    rows, cols = [2, 3], [4, 1]
    C, C_p = 3, 5
    s_row, s_col = rng.standard_normal((5, C)), rng.standard_normal((5, C))
    Wa, Wb = rng.standard_normal((C_p, C)), rng.standard_normal((C_p, C))
    z = pair_broadcast_rect(rows, cols, s_row, s_col, Wa, Wb)
    tR, tC, ta, tb = (torch.from_numpy(x) for x in (s_row, s_col, Wa, Wb))
    cell, r0, c0 = 0, 0, 0
    for n, m in zip(rows, cols):
        for a in range(n):
            for b in range(m):
                ref = F.linear(tR[r0 + a], ta) + F.linear(tC[c0 + b], tb)
                assert np.allclose(z[cell], ref.numpy(), rtol=1e-13, atol=1e-13)
                cell += 1
        r0 += n
        c0 += m


def pin_rect_reduce_closed_form(pair_broadcast_rect, pair_reduce_rect, rng):
    """Without a transition, (1/M_i) sum_b (U[a] + V[b]) = U[a] + mean of the
    sample's M_i column projections; M_i = 0 gives zero rows."""
    rows, cols = [3, 2, 4, 1], [5, 1, 2, 0]
    C, C_p = 4, 3
    s_row = rng.standard_normal((sum(rows), C))
    s_col = rng.standard_normal((sum(cols), C))
    Wa, Wb = rng.standard_normal((C_p, C)), rng.standard_normal((C_p, C))
    z = pair_broadcast_rect(rows, cols, s_row, s_col, Wa, Wb)
    m, _ = pair_reduce_rect(rows, cols, z)
    U, V = s_row @ Wa.T, s_col @ Wb.T
    r0, c0 = 0, 0
    for n, mm in zip(rows, cols):
        for a in range(n):
            ref = U[r0 + a] + V[c0:c0 + mm].sum(axis=0) / mm if mm else np.zeros(C_p)
            assert np.allclose(m[r0 + a], ref, rtol=1e-12, atol=1e-12)
        r0 += n
        c0 += mm


# ----------------------------------------------------------------------------
# SwiGLU transition ("DanLing NestedTensor" Eq. 1, h is a SwiGLU update)
# ----------------------------------------------------------------------------

def pin_silu(silu):
    """SiLU(0) = 0; SiLU(x) - SiLU(-x) = x for every x; SiLU(x) -> x for
    large x and -> 0 for large negative x."""
    x = np.linspace(-30, 30, 121)
    y = silu(x)
    assert silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(y - silu(-x), x, rtol=1e-14, atol=1e-13)
    assert abs(silu(np.array([40.0]))[0] - 40.0) < 1e-12 and abs(silu(np.array([-40.0]))[0]) < 1e-12


def pin_swiglu_library(transition_swiglu, rng, biases=True):
    """LN -> (SiLU(gate) * value) -> Linear plus residual equals
    torch.nn.functional's layer_norm / linear / silu in float64."""
    P, C_p, H = 29, 8, 32
    z = rng.standard_normal((P, C_p)) * 2.0 - 0.3
    gamma = 1.0 + 0.1 * rng.standard_normal(C_p)
    beta = 0.1 * rng.standard_normal(C_p)
    W1, W3, W2 = rng.standard_normal((H, C_p)), rng.standard_normal((H, C_p)), rng.standard_normal((C_p, H))
    b1, b3, b2 = (rng.standard_normal(n) if biases else None for n in (H, H, C_p))
    got = transition_swiglu(z, gamma, beta, 1e-5, W1, b1, W3, b3, W2, b2)
    t = lambda a: None if a is None else torch.from_numpy(a)
    ln = F.layer_norm(t(z), (C_p,), t(gamma), t(beta), 1e-5)
    hid = F.silu(F.linear(ln, t(W1), t(b1))) * F.linear(ln, t(W3), t(b3))
    ref = t(z) + F.linear(hid, t(W2), t(b2))
    assert np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def pin_swiglu_zero_gate(transition_swiglu, rng):
    """A zero gate (W1 = 0, b1 = 0) closes the update: SiLU(0) = 0, so
    z~ = z + b2 exactly, whatever W3 and W2 are."""
    z = rng.standard_normal((9, 6))
    b2 = rng.standard_normal(6)
    out = transition_swiglu(z, np.ones(6), np.zeros(6), 1e-5, np.zeros((12, 6)), None,
                            rng.standard_normal((12, 6)), rng.standard_normal(12), rng.standard_normal((6, 12)), b2)
    assert np.array_equal(out, z + b2)


def pin_attention_backward_autograd(varlen_attention_backward, rng):
    """Per segment, the gradients equal torch autograd of SDPA in float64
    (non-causal and causal, equal and differing query/key lengths)."""
    cu_q, cu_k = [0, 5, 5, 12, 14], [0, 7, 9, 16, 16]
    H, d = 2, 4
    q = rng.standard_normal((cu_q[-1], H, d))
    do = rng.standard_normal((cu_q[-1], H, d))
    k, v = (rng.standard_normal((cu_k[-1], H, d)) for _ in range(2))
    for causal in (False, True):
        for ck in (None, cu_k):
            if ck is None:                        # self-attention: keys share the query offsets
                kk, vv, cuk = k[:cu_q[-1]], v[:cu_q[-1]], cu_q
            else:
                kk, vv, cuk = k, v, cu_k
            dq, dk, dv = varlen_attention_backward(q, kk, vv, do, cu_q, causal=causal, cu_seqlens_k=ck)
            for b in range(len(cu_q) - 1):
                ql, qh, kl, kh = cu_q[b], cu_q[b + 1], cuk[b], cuk[b + 1]
                if qh == ql or kh == kl:
                    assert np.all(dq[ql:qh] == 0)
                    continue
                tq = torch.tensor(q[ql:qh].transpose(1, 0, 2), requires_grad=True)
                tk = torch.tensor(kk[kl:kh].transpose(1, 0, 2), requires_grad=True)
                tv = torch.tensor(vv[kl:kh].transpose(1, 0, 2), requires_grad=True)
                mask = None
                if causal:
                    mask = torch.ones(qh - ql, kh - kl, dtype=torch.bool).tril(kh - kl - (qh - ql))
                    if not mask.any(dim=1).all():
                        continue          # rows with no key: SDPA gives NaN there; covered elsewhere
                out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
                out.backward(torch.from_numpy(do[ql:qh].transpose(1, 0, 2)))
                assert np.allclose(dq[ql:qh], tq.grad.numpy().transpose(1, 0, 2), rtol=1e-10, atol=1e-10)
                assert np.allclose(dk[kl:kh], tk.grad.numpy().transpose(1, 0, 2), rtol=1e-10, atol=1e-10)
                assert np.allclose(dv[kl:kh], tv.grad.numpy().transpose(1, 0, 2), rtol=1e-10, atol=1e-10)


# ----------------------------------------------------------------------------
# Eq. 5 loss and the block's gradients ("DanLing NestedTensor" Appendix A.1,
# Eq. 5; the chain rule of Eq. 1)
# ----------------------------------------------------------------------------

def pin_eq5_weights(eq5_sample_weights):
    """alpha_i = 1 + i/B and beta_i = 1.5 - i/(2B), evaluated by hand for B = 4."""
    a, b = eq5_sample_weights(4)
    assert np.allclose(a, [1.0, 1.25, 1.5, 1.75], rtol=0, atol=1e-15)
    assert np.allclose(b, [1.5, 1.375, 1.25, 1.125], rtol=0, atol=1e-15)


def pin_eq5_closed_form(eq5_loss):
    """All-ones outputs: L = sum_i alpha_i N_i / T + sum_i beta_i N_i^2 / P
    (C and C_p cancel); doubling both outputs multiplies L by four; an
    output of zeros contributes nothing."""
    lengths = [3, 0, 2, 5]
    T, P = 10, 9 + 4 + 25
    a = [1.0, 1.25, 1.5, 1.75]
    b = [1.5, 1.375, 1.25, 1.125]
    s_out = np.ones((T, 6))
    z = np.ones((P, 4))
    want = (a[0] * 3 + a[2] * 2 + a[3] * 5) / T + (b[0] * 9 + b[2] * 4 + b[3] * 25) / P
    assert abs(eq5_loss(lengths, s_out, z) - want) < 1e-12
    assert abs(eq5_loss(lengths, 2 * s_out, 2 * z) - 4 * want) < 1e-12
    assert abs(eq5_loss(lengths, 0 * s_out, z) - (b[0] * 9 + b[2] * 4 + b[3] * 25) / P) < 1e-12


def _torch_block_eq5(lengths, s, W, with_bias):
    """Eq. 1 per sample and Eq. 5 in torch float64 (F.linear, F.layer_norm,
    relu, mean over the column axis), for autograd."""
    B = len(lengths)
    C, C_p = s.shape[1], W["W_a"].shape[0]
    T = sum(lengths)
    P = sum(n * n for n in lengths)
    lx = s.new_zeros(())
    lp = s.new_zeros(())
    off = 0
    for i, n in enumerate(lengths):
        if n == 0:
            continue
        X = s[off:off + n]
        off += n
        pair = F.linear(X, W["W_a"])[:, None, :] + F.linear(X, W["W_b"])[None, :, :]
        y = F.layer_norm(pair, (C_p,), W["gamma"], W["beta"], eps=1e-5)
        upd = F.linear(torch.relu(F.linear(y, W["W1"], W["b1"] if with_bias else None)), W["W2"],
                       W["b2"] if with_bias else None)
        pt = pair + upd
        xt = X + F.linear(pt.mean(dim=1), W["W_g"], W["b_g"] if with_bias else None)
        lx = lx + (1 + i / B) * (xt ** 2).sum()
        lp = lp + (1.5 - i / (2 * B)) * (pt ** 2).sum()
    return lx / (C * T) + lp / (C_p * P)


def _block_problem(rng, lengths, C=6, C_p=4, H=8, with_bias=True):
    from oracle.block import Weights
    T = sum(lengths)
    s = rng.standard_normal((T, C))
    W = {"W_a": rng.standard_normal((C_p, C)) / np.sqrt(C), "W_b": rng.standard_normal((C_p, C)) / np.sqrt(C),
         "gamma": 1 + 0.3 * rng.standard_normal(C_p), "beta": 0.2 * rng.standard_normal(C_p),
         "W1": rng.standard_normal((H, C_p)) / 2, "b1": 0.3 * rng.standard_normal(H),
         "W2": rng.standard_normal((C_p, H)) / 3, "b2": 0.2 * rng.standard_normal(C_p),
         "W_g": rng.standard_normal((C, C_p)) / 2, "b_g": 0.1 * rng.standard_normal(C)}
    if not with_bias:
        W["b1"] = W["b2"] = W["b_g"] = None
    w = Weights(W["W_a"], W["W_b"], W["gamma"], W["beta"], 1e-5, W["W1"], W["b1"], W["W2"], W["b2"], W["W_g"],
                W["b_g"])
    return s, W, w


def pin_block_backward_autograd(block_loss_and_grads, block_packed, rng):
    """The loss and every gradient equal torch autograd of an independent
    torch formulation of Eq. 1 + Eq. 5 in float64 (zero-length samples
    included, with and without biases)."""
    for lengths, with_bias in (([3, 0, 4, 1], True), ([5, 2], False)):
        s, W, w = _block_problem(rng, lengths, with_bias=with_bias)
        fwd = block_packed(lengths, s, w)
        loss, g = block_loss_and_grads(lengths, s, w, fwd.z_tilde, fwd.s_out)
        ts = torch.tensor(s, requires_grad=True)
        tW = {k: (None if v is None else torch.tensor(v, requires_grad=True)) for k, v in W.items()}
        tl = _torch_block_eq5(lengths, ts, tW, with_bias)
        tl.backward()
        tlf = float(tl.detach())
        assert abs(loss - tlf) < 1e-12 * max(1.0, abs(tlf))
        pairs = [("ds", ts), ("dW_a", tW["W_a"]), ("dW_b", tW["W_b"]), ("dgamma", tW["gamma"]),
                 ("dbeta", tW["beta"]), ("dW1", tW["W1"]), ("dW2", tW["W2"]), ("dW_g", tW["W_g"])]
        if with_bias:
            pairs += [("db1", tW["b1"]), ("db2", tW["b2"]), ("db_g", tW["b_g"])]
        for name, t in pairs:
            got = getattr(g, name)
            assert got.shape == tuple(t.grad.shape), name
            assert np.allclose(got, t.grad.numpy(), rtol=1e-9, atol=1e-12), name


def pin_block_backward_finite_differences(block_loss_and_grads, block_packed, rng):
    """Central differences of the loss (through the oracle's own forward)
    match the gradient on a few coordinates of the singles and weights."""
    from oracle.block_backward import eq5_loss
    lengths = [2, 3]
    s, W, w = _block_problem(rng, lengths)
    fwd = block_packed(lengths, s, w)
    _, g = block_loss_and_grads(lengths, s, w, fwd.z_tilde, fwd.s_out)

    def loss_at(s_, w_):
        f = block_packed(lengths, s_, w_)
        return eq5_loss(lengths, f.s_out, f.z_tilde)

    h = 1e-6
    for name, idx in (("ds", (1, 2)), ("dW1", (3, 1)), ("dW_a", (2, 4)), ("dgamma", (1,)), ("dW_g", (0, 3)),
                      ("db2", (2,))):
        if name == "ds":
            sp, sm = s.copy(), s.copy()
            sp[idx] += h
            sm[idx] -= h
            fd = (loss_at(sp, w) - loss_at(sm, w)) / (2 * h)
        else:
            attr = {"dW1": "W1", "dW_a": "W_a", "dgamma": "gamma", "dW_g": "W_g", "db2": "b2"}[name]
            arr = getattr(w, attr)
            old = arr[idx]
            arr[idx] = old + h
            lp_ = loss_at(s, w)
            arr[idx] = old - h
            lm_ = loss_at(s, w)
            arr[idx] = old
            fd = (lp_ - lm_) / (2 * h)
        assert abs(fd - getattr(g, name)[idx]) < 1e-6 * max(1.0, abs(fd)), name
