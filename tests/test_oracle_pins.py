"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import numpy as np
import pytest

import _pins as pins
from _helpers import oracle_weights, f64
from oracle import partition as opart
from oracle import block as oblock
from oracle import attention as oattn
from variable_length_batching_gb300 import workloads as wl


def rng(seed=0):
    return np.random.default_rng(seed)


def test_fig2_worked_example():
    pins.pin_fig2(opart.partition)


@pytest.mark.parametrize("lengths", [[2, 3], [0], [5, 0, 0, 3], [1] * 7, [0, 0], list(range(9, 0, -1))])
def test_partition_invariants_and_bruteforce(lengths):
    pins.pin_partition_invariants(opart.partition, lengths)
    pins.pin_partition_bruteforce(opart.partition, lengths)


def test_partition_random():
    r = rng(3)
    for _ in range(20):
        lengths = list(r.integers(0, 12, size=r.integers(1, 9)))
        pins.pin_partition_invariants(opart.partition, lengths)
        pins.pin_partition_bruteforce(opart.partition, lengths)


def test_partition_rejects_negative():
    with pytest.raises(ValueError):
        opart.partition([3, -1])


def test_compatibility_same_rows_different_partition():
    """Equal totals do not make partitions equal (section 3.2 'Compatibility
    and semantics'): (3, 4) and (5, 0) both hold 25 pair cells."""
    a, b = opart.partition([3, 4]), opart.partition([5, 0])
    assert a.P == b.P == 25
    assert (a.T, list(a.row_start)) != (b.T, list(b.row_start))


def test_pair_storage_is_sum_of_squares():
    """Packed pair storage is sum_i N_i^2 rows against B * N_max^2 padded
    (abstract; section 1)."""
    assert opart.partition([2, 3]).P == 13 and opart.padded_cells([2, 3]) == 18
    for cfg in wl.BLOCK_CONFIGS.values():
        lengths = wl.draw_lengths(cfg, np.random.default_rng(cfg.seed))
        p = opart.partition(lengths)
        assert p.P == int((lengths.astype(np.int64) ** 2).sum())
        assert opart.padded_cells(lengths) == cfg.B * int(lengths.max()) ** 2
        assert p.P <= opart.padded_cells(lengths)


def test_broadcast_onehot():
    pins.pin_broadcast_onehot(oblock.pair_broadcast, rng(1))


def test_broadcast_left_right():
    pins.pin_broadcast_left_right(oblock.pair_broadcast, rng(2))


@pytest.mark.parametrize("biases", [True, False])
def test_transition_matches_torch(biases):
    pins.pin_transition_library(oblock.pair_transition, rng(4), biases)


def test_transition_identity():
    pins.pin_transition_identity(oblock.pair_transition, rng(5))


def test_layernorm_constant():
    pins.pin_layernorm_constant(oblock.layer_norm, rng(6))


def test_reduce_closed_form():
    pins.pin_reduce_closed_form(oblock.pair_broadcast, oblock.pair_reduce, rng(7))


def test_reduce_invariants():
    pins.pin_reduce_invariants(oblock.pair_reduce, rng(8))


def test_reduce_bruteforce():
    pins.pin_reduce_bruteforce(oblock.pair_reduce, rng(9))


@pytest.mark.parametrize("lengths", [[5, 2, 7], [1, 6], [4, 0, 3]])
def test_packed_equals_padded(lengths):
    cfg = wl.TINY_FP32
    inp = wl.make_block_inputs(cfg, lengths=lengths, biases=True, seed=11)
    w = oracle_weights(inp.blocks[0])
    pins.pin_packed_equals_padded(oblock.block_packed, oblock.block_padded_gathered, w, lengths, f64(inp.s))


def test_block_steps_compose():
    """The call-boundary functions chained reproduce the dense per-sample block."""
    cfg = wl.TINY_FP32
    inp = wl.make_block_inputs(cfg, biases=True)
    w = oracle_weights(inp.blocks[0])
    s = f64(inp.s)
    L = inp.lengths
    full = oblock.block_packed(L, s, w)
    z = oblock.pair_broadcast(L, s, s, w.W_a, w.W_b)
    zt = oblock.pair_transition(z, w.gamma, w.beta, w.eps, w.W1, w.b1, w.W2, w.b2)
    m, s_out = oblock.pair_reduce(L, zt, w.W_g, w.b_g, s)
    assert np.allclose(z, full.z, rtol=1e-13, atol=1e-13)
    assert np.allclose(zt, full.z_tilde, rtol=1e-12, atol=1e-12)
    assert np.allclose(m, full.m, rtol=1e-12, atol=1e-12)
    assert np.allclose(s_out, full.s_out, rtol=1e-12, atol=1e-12)


def test_sampled_evaluation_matches_full():
    cfg = wl.TINY_FP32
    inp = wl.make_block_inputs(cfg, biases=True)
    w = oracle_weights(inp.blocks[0])
    s = f64(inp.s)
    full = oblock.block_packed(inp.lengths, s, w)
    cells = np.random.default_rng(0).integers(0, full.z.shape[0], size=50)
    P, Pt = oblock.block_cells(inp.lengths, s, w, cells)
    assert np.allclose(P, full.z[cells], rtol=1e-12, atol=1e-12)
    assert np.allclose(Pt, full.z_tilde[cells], rtol=1e-12, atol=1e-12)
    rows = [0, 5, 28, 29, 85]
    m, so = oblock.block_rows(inp.lengths, s, w, rows)
    assert np.allclose(m, full.m[rows], rtol=1e-12, atol=1e-12)
    assert np.allclose(so, full.s_out[rows], rtol=1e-12, atol=1e-12)


def test_g_identity_adds_mean():
    """With C = C_p, W_g = I and no bias, X~ = X + m."""
    lengths = [3, 2]
    r = rng(12)
    C = 4
    s = r.standard_normal((5, C))
    w = oblock.Weights(W_a=r.standard_normal((C, C)), W_b=r.standard_normal((C, C)), gamma=np.ones(C),
                       beta=np.zeros(C), eps=1e-5, W1=r.standard_normal((8, C)), b1=None,
                       W2=r.standard_normal((C, 8)), b2=None, W_g=np.eye(C), b_g=None)
    out = oblock.block_packed(lengths, s, w)
    assert np.allclose(out.s_out, s + out.m, rtol=1e-14, atol=1e-14)


def test_stacked_blocks_chain_singles():
    cfg = wl.TINY_FP32
    inp = wl.make_block_inputs(cfg)
    w = oracle_weights(inp.blocks[0])
    s = f64(inp.s)
    x2, last = oblock.stacked_blocks(inp.lengths, s, [w, w])
    once = oblock.block_packed(inp.lengths, s, w)
    twice = oblock.block_packed(inp.lengths, once.s_out, w)
    assert np.array_equal(x2, twice.s_out) and np.array_equal(last.z_tilde, twice.z_tilde)


def test_attention_single_segment_sdpa():
    pins.pin_attention_single_segment_sdpa(oattn.varlen_attention, rng(13))


def test_attention_masked_core_math():
    pins.pin_attention_masked_core_math(oattn.masked_full_attention, rng(14))


def test_attention_varlen_equals_masked():
    pins.pin_attention_varlen_equals_masked(oattn.varlen_attention, oattn.masked_full_attention, rng(15))


def test_attention_special_cases():
    pins.pin_attention_special_cases(oattn.varlen_attention, rng(16))


def test_attention_flops_config():
    lens = wl.draw_segments(65536, 16, 512, np.random.default_rng(0))
    assert len(lens) == 237 and int(lens.sum()) == 65536
    assert int((lens.astype(np.int64) ** 2).sum()) == 23342596
    assert oattn.attention_flops(lens, 12, 64) == 4 * 23342596 * 12 * 64


def test_attention_causal_sdpa():
    pins.pin_attention_causal_sdpa(oattn.varlen_attention, rng(17))


def test_attention_cross_sdpa():
    pins.pin_attention_cross_sdpa(oattn.varlen_attention, rng(18))


def test_attention_causal_masked():
    pins.pin_attention_causal_masked(oattn.varlen_attention, oattn.masked_full_attention_causal, rng(19))


def test_rect_partition_bruteforce():
    from oracle import partition as op
    pins.pin_rect_partition_bruteforce(op.partition_rect, [2, 0, 3, 1, 4], [3, 2, 0, 1, 4])
    r = rng(20)
    for _ in range(20):
        B = int(r.integers(0, 7))
        pins.pin_rect_partition_bruteforce(op.partition_rect, list(r.integers(0, 9, B)), list(r.integers(0, 9, B)))


def test_rect_square_case():
    from oracle import partition as op
    pins.pin_rect_square_case(op.partition_rect, op.partition, [2, 3, 0, 5])


def test_rect_broadcast_onehot():
    pins.pin_rect_broadcast_onehot(oblock.pair_broadcast_rect, rng(21))


def test_rect_broadcast_library():
    pins.pin_rect_broadcast_library(oblock.pair_broadcast_rect, rng(22))


def test_rect_reduce_closed_form():
    pins.pin_rect_reduce_closed_form(oblock.pair_broadcast_rect, oblock.pair_reduce_rect, rng(23))


def test_rect_block_square_case_equals_square_block():
    """The rectangular block with Z = X and M_i = N_i is the square block."""
    r = rng(24)
    lengths = [3, 1, 4]
    C, C_p, H = 6, 4, 8
    s = r.standard_normal((sum(lengths), C))
    w = oblock.Weights(W_a=r.standard_normal((C_p, C)), W_b=r.standard_normal((C_p, C)),
                       gamma=1 + 0.1 * r.standard_normal(C_p), beta=0.1 * r.standard_normal(C_p), eps=1e-5,
                       W1=r.standard_normal((H, C_p)), b1=r.standard_normal(H), W2=r.standard_normal((C_p, H)),
                       b2=r.standard_normal(C_p), W_g=r.standard_normal((C, C_p)), b_g=r.standard_normal(C))
    a = oblock.block_packed_rect(lengths, lengths, s, s, w)
    b = oblock.block_packed(lengths, s, w)
    for x, y in ((a.z, b.z), (a.z_tilde, b.z_tilde), (a.m, b.m), (a.s_out, b.s_out)):
        assert np.allclose(x, y, rtol=1e-13, atol=1e-13)


def test_silu():
    pins.pin_silu(oblock.silu)


def test_swiglu_library():
    pins.pin_swiglu_library(oblock.transition_swiglu, rng(25))
    pins.pin_swiglu_library(oblock.transition_swiglu, rng(26), biases=False)


def test_swiglu_zero_gate():
    pins.pin_swiglu_zero_gate(oblock.transition_swiglu, rng(27))


def test_attention_backward_autograd():
    pins.pin_attention_backward_autograd(oattn.varlen_attention_backward, rng(28))
