"""GPU parity: every library call against the CPU oracle on the same seeded
inputs.  Partitions are compared bit for bit; floats normwise,
max|gpu - oracle| / max|oracle| <= 2e-2 (bf16 I/O, fp32 accumulation) or
1e-5 (fp32 mode), per output tensor."""
import ctypes
from types import SimpleNamespace

import numpy as np
import pytest
import torch

from _helpers import TOL, f64, normwise_err, oracle_weights, to_np
from oracle import attention as oattn
from oracle import block as oblock
from oracle import partition as opart
from variable_length_batching_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def nt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_batching_gb300 import build, nt as ntmod
    build.build()
    return ntmod


def dev_weights(w: wl.BlockWeights):
    g = lambda t: None if t is None else t.to(DEV).contiguous()
    return SimpleNamespace(W_a=g(w.W_a), W_b=g(w.W_b), ln_gamma=g(w.ln_gamma), ln_beta=g(w.ln_beta),
                           W1=g(w.W1), b1=g(w.b1), W2=g(w.W2), b2=g(w.b2), W_g=g(w.W_g), b_g=g(w.b_g))


def dev_lengths(lengths):
    return torch.as_tensor(np.asarray(lengths, dtype=np.int32)).to(DEV)


# ----------------------------------------------------------------------------
# a1 partitions: bit-exact
# ----------------------------------------------------------------------------

PARTITION_CASES = [
    [2, 3],                       # Figure 2
    [0], [1], [5, 0, 0, 3, 0], [1] * 33, [1024],
    list(range(1, 2049)),         # B > 1024: the scan carries across chunks
]


@pytest.mark.parametrize("lengths", PARTITION_CASES + [list(wl.draw_lengths(c, np.random.default_rng(0)))
                                                      for c in wl.BLOCK_CONFIGS.values()])
def test_partition_bit_exact(nt, lengths):
    part = nt.nt_partition_build(dev_lengths(lengths))
    ref = opart.partition(lengths)
    assert (part.T, part.P, part.max_len) == (ref.T, ref.P, ref.max_len)
    assert np.array_equal(part.cu_seqlens.cpu().numpy(), ref.cu_seqlens)
    assert np.array_equal(part.pair_off.cpu().numpy(), ref.pair_off)
    assert np.array_equal(part.row_start.cpu().numpy(), ref.row_start)
    if ref.T:
        assert np.array_equal(part.row_sample[: ref.T].cpu().numpy(), ref.row_sample)
    nt.nt_device_status()


@pytest.mark.parametrize("lengths", [[3, 0, 5, 1, 130, 7], [0, 0], [4], list(range(1, 200))])
def test_partition_with_rows_matches_two_calls(nt, lengths):
    """nt_partition_build_with_rows (row splits after the scan in the stream,
    T and P from the device totals) equals the two-call partition bit for
    bit, with an exact capacity and with a larger one."""
    ref = nt.nt_partition_build(dev_lengths(lengths))
    T = int(sum(lengths))
    for cap in (T, T + 37):
        got = nt.nt_partition_build(dev_lengths(lengths), T=cap)
        assert (got.T, got.P, got.max_len) == (ref.T, ref.P, ref.max_len)
        for a, b in ((got.cu_seqlens, ref.cu_seqlens), (got.pair_off, ref.pair_off)):
            assert torch.equal(a, b)
        assert torch.equal(got.row_start[:T + 1], ref.row_start)
        if T:
            assert torch.equal(got.row_sample[:T], ref.row_sample[:T])
    nt.nt_device_status()


# one-launch partitions (1 <= B <= 1024, capacity <= 65,536) and the scan +
# row-split pair beyond either bound, each at its edge
WITH_ROWS_CASES = [
    ([2, 3], None), ([0, 0, 5, 0], None), ([7, 0], None), ([1] * 1024, None), ([1] * 1025, None),
    ([256] * 256, None), ([256] * 256, 65537), ([300] * 10, 70000), (list(range(0, 300, 3)), None),
]


@pytest.mark.parametrize("lengths,cap", WITH_ROWS_CASES)
def test_partition_with_rows_bit_exact(nt, lengths, cap):
    """nt_partition_build_with_rows against the oracle's partition, bit for
    bit, on both kernel paths."""
    ref = opart.partition(lengths)
    part = nt.nt_partition_build(dev_lengths(lengths), T=ref.T if cap is None else cap)
    assert (part.T, part.P, part.max_len) == (ref.T, ref.P, ref.max_len)
    assert np.array_equal(part.cu_seqlens.cpu().numpy(), ref.cu_seqlens)
    assert np.array_equal(part.pair_off.cpu().numpy(), ref.pair_off)
    assert np.array_equal(part.row_start[: ref.T + 1].cpu().numpy(), ref.row_start)
    if ref.T:
        assert np.array_equal(part.row_sample[: ref.T].cpu().numpy(), ref.row_sample)
    nt.nt_device_status()


@pytest.mark.parametrize("lengths,cap", [([64, 100, 3], 50), ([2] * 1100, 2000)])
def test_partition_with_rows_small_capacity_rejected(nt, lengths, cap):
    """A capacity below the lengths' sum is reported (NT_ERR_INVALID) after
    the totals come back; the row splits write nothing past the buffers they
    were given (one-launch path, then the scan + row-split pair)."""
    B = len(lengths)
    guard = torch.full((64,), -7, dtype=torch.int64, device=DEV)
    buf = torch.empty(cap + 1 + 64, dtype=torch.int64, device=DEV)
    buf[cap + 1:] = guard
    rs_guard = torch.full((64,), -9, dtype=torch.int32, device=DEV)
    rs = torch.empty(cap + 64, dtype=torch.int32, device=DEV)
    rs[cap:] = rs_guard
    with pytest.raises(nt.NTError) as ei:
        c = nt.nt_partition()
        L = dev_lengths(lengths)
        cu = torch.empty(B + 1, dtype=torch.int32, device=DEV)
        po = torch.empty(B + 1, dtype=torch.int64, device=DEV)
        tot = torch.empty(4, dtype=torch.int64, device=DEV)
        st = nt.lib().nt_partition_build_with_rows(nt._ptr(L), B, cap, nt._ptr(cu), nt._ptr(po), nt._ptr(tot),
                                                   nt._ptr(buf), nt._ptr(rs), ctypes.byref(c), nt._stream(None))
        nt._check(st, "nt_partition_build_with_rows")
    assert ei.value.status == 1
    assert torch.equal(buf[cap + 1:], guard)     # nothing written past row_start's cap + 1 entries
    assert torch.equal(rs[cap:], rs_guard)       # nor past row_sample's cap entries
    ref = opart.partition(lengths)
    assert np.array_equal(buf[:cap].cpu().numpy(), ref.row_start[:cap])   # the rows that fit are right
    nt.nt_device_status()


def test_partition_empty_batch(nt):
    part = nt.nt_partition_build(torch.empty(0, dtype=torch.int32, device=DEV))
    assert (part.B, part.T, part.P) == (0, 0, 0)
    assert part.cu_seqlens.cpu().tolist() == [0] and part.row_start.cpu().tolist() == [0]


def test_partition_negative_length_rejected(nt):
    with pytest.raises(nt.NTError) as ei:
        nt.nt_partition_build(dev_lengths([3, -2, 4]))
    assert ei.value.status == 1


# ----------------------------------------------------------------------------
# a2-a4 one call at a time, inputs straight from the seeded generators
# ----------------------------------------------------------------------------

# bf16 widths other than the bench's: the u, v projections at N = C_z = 64
# (one 64-column tile) and g at N = C_s = 192 (three) with K = 64 and 192
NARROW_BF16 = wl.BlockConfig("narrow_bf16_B5_N8-150_Cs192_Cz64", B=5, length_rule="uniform", rule_args=(8, 150),
                             C_s=192, C_z=64, H_t=256, dtype=wl.BF16)

STEP_CASES = [
    (wl.TINY_FP32, None),
    (wl.PAIRFORMER_BF16, None),
    (wl.PAIRFORMER_BF16, [0, 1, 7, 0, 130, 2, 1, 33]),   # zero and unit lengths, ragged tails
    (wl.TINY_FP32, [0, 9, 1, 0, 31, 3]),
    (NARROW_BF16, None),
    (NARROW_BF16, [0, 9, 150, 1, 77, 130]),
]


@pytest.mark.parametrize("cfg,lengths", STEP_CASES)
def test_broadcast(nt, cfg, lengths):
    inp = wl.make_block_inputs(cfg, lengths=lengths)
    w = inp.blocks[0]
    part = nt.nt_partition_build(dev_lengths(inp.lengths))
    s = inp.s.to(DEV)
    z = nt.nt_pair_broadcast(part, s, s, w.W_a.to(DEV), w.W_b.to(DEV))
    ref = oblock.pair_broadcast(inp.lengths, f64(inp.s), f64(inp.s), f64(w.W_a), f64(w.W_b))
    assert z.shape == ref.shape
    assert normwise_err(to_np(z), ref, dtype=cfg.dtype) <= TOL[cfg.dtype]
    nt.nt_device_status()


def test_broadcast_left_right_distinct(nt):
    cfg = wl.PAIRFORMER_BF16
    inp = wl.make_block_inputs(cfg, lengths=[17, 64, 3])
    w = inp.blocks[0]
    sR = wl.random_rows(inp.s.shape[0], cfg.C_s, cfg.dtype, seed=5)
    part = nt.nt_partition_build(dev_lengths(inp.lengths))
    z = nt.nt_pair_broadcast(part, inp.s.to(DEV), sR.to(DEV), w.W_a.to(DEV), w.W_b.to(DEV))
    ref = oblock.pair_broadcast(inp.lengths, f64(inp.s), f64(sR), f64(w.W_a), f64(w.W_b))
    assert normwise_err(to_np(z), ref, dtype=cfg.dtype) <= TOL[cfg.dtype]


@pytest.mark.parametrize("cfg,rows,biases", [(wl.TINY_FP32, 1966, False), (wl.TINY_FP32, 517, True),
                                             (wl.PAIRFORMER_BF16, 20000, False),
                                             (wl.PAIRFORMER_BF16, 4099, True),
                                             (wl.PAIRFORMER_BF16, 1, True)])
def test_transition(nt, cfg, rows, biases):
    inp = wl.make_block_inputs(cfg, lengths=[1], biases=biases)
    w = inp.blocks[0]
    z = wl.random_rows(rows, cfg.C_z, cfg.dtype, seed=rows, scale=1.5)
    part = nt.nt_partition_build(dev_lengths([1] * rows))   # rows one-cell samples: P = rows
    wd = dev_weights(w)
    zd = z.to(DEV)
    out = nt.nt_pair_transition(part, zd, wd.ln_gamma, wd.ln_beta, wd.W1, wd.b1, wd.W2, wd.b2)
    ref = oblock.pair_transition(f64(z), f64(w.ln_gamma), f64(w.ln_beta), 1e-5, f64(w.W1), f64(w.b1),
                                 f64(w.W2), f64(w.b2))
    assert normwise_err(to_np(out), ref, dtype=cfg.dtype) <= TOL[cfg.dtype]
    # in place gives the same bits
    nt.nt_pair_transition(part, zd, wd.ln_gamma, wd.ln_beta, wd.W1, wd.b1, wd.W2, wd.b2, out=zd)
    assert torch.equal(zd, out)
    nt.nt_device_status()


@pytest.mark.parametrize("cfg,lengths", STEP_CASES)
def test_reduce(nt, cfg, lengths):
    inp = wl.make_block_inputs(cfg, lengths=lengths, biases=True)
    w = inp.blocks[0]
    ref_part = opart.partition(inp.lengths)
    z = wl.random_rows(ref_part.P, cfg.C_z, cfg.dtype, seed=3)
    part = nt.nt_partition_build(dev_lengths(inp.lengths))
    s = inp.s.to(DEV)
    m, s_out = nt.nt_pair_reduce(part, z.to(DEV), w.W_g.to(DEV), w.b_g.to(DEV), s_in=s)
    m_ref, s_ref = oblock.pair_reduce(inp.lengths, f64(z), f64(w.W_g), f64(w.b_g), f64(inp.s))
    assert normwise_err(to_np(m), m_ref, dtype=cfg.dtype) <= TOL[cfg.dtype]
    assert normwise_err(to_np(s_out), s_ref, dtype=cfg.dtype) <= TOL[cfg.dtype]
    m2, none = nt.nt_pair_reduce(part, z.to(DEV))
    assert none is None and torch.equal(m2, m)


# ----------------------------------------------------------------------------
# The whole block, chained through the library, against the dense oracle
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("cfg,lengths,biases", [(wl.TINY_FP32, None, False), (wl.TINY_FP32, None, True),
                                                (wl.PAIRFORMER_BF16, None, False),
                                                (wl.PAIRFORMER_BF16, [0, 1, 7, 0, 130, 2, 1, 33], True)])
def test_block_full(nt, cfg, lengths, biases):
    inp = wl.make_block_inputs(cfg, lengths=lengths, biases=biases)
    w = inp.blocks[0]
    part = nt.nt_partition_build(dev_lengths(inp.lengths))
    z, m, s_out = nt.block_forward(part, inp.s.to(DEV), dev_weights(w))
    ref = oblock.block_packed(inp.lengths, f64(inp.s), oracle_weights(w))
    tol = TOL[cfg.dtype]
    assert normwise_err(to_np(z), ref.z_tilde, dtype=cfg.dtype) <= tol
    assert normwise_err(to_np(m), ref.m, dtype=cfg.dtype) <= tol
    assert normwise_err(to_np(s_out), ref.s_out, dtype=cfg.dtype) <= tol
    nt.nt_device_status()


@pytest.mark.parametrize("cfg", [wl.LOGNORMAL_BF16, wl.NEAR_UNIFORM_BF16, wl.STACKED4_BF16])
def test_block_full_size_sampled(nt, cfg):
    """Full-size workloads, first block: sampled cells and rows, each computed
    one by one by the oracle from its definition.  Also checks the packed
    pair storage is exactly sum N_i^2 rows (never B * N_max^2)."""
    inp = wl.make_block_inputs(cfg)
    part = nt.nt_partition_build(dev_lengths(inp.lengths))
    ref_part = opart.partition(inp.lengths)
    assert part.P == ref_part.P < opart.padded_cells(inp.lengths)
    w = inp.blocks[0]
    z, m, s_out = nt.block_forward(part, inp.s.to(DEV), dev_weights(w))
    assert z.shape == (ref_part.P, cfg.C_z)
    ow = oracle_weights(w)
    rng = np.random.default_rng(1)
    cells = np.concatenate([rng.integers(0, ref_part.P, size=1500), ref_part.pair_off[1:-1] - 1,
                            ref_part.pair_off[:-1], [ref_part.P - 1]])
    _, Pt = oblock.block_cells(inp.lengths, f64(inp.s), ow, cells)
    got = to_np(z[torch.as_tensor(cells, device=DEV)])
    assert normwise_err(got, Pt, dtype=cfg.dtype) <= TOL[cfg.dtype]
    rows = np.concatenate([rng.integers(0, ref_part.T, size=12), ref_part.cu_seqlens[:-1]])
    m_ref, s_ref = oblock.block_rows(inp.lengths, f64(inp.s), ow, rows)
    idx = torch.as_tensor(rows, device=DEV)
    assert normwise_err(to_np(m[idx]), m_ref, dtype=cfg.dtype) <= TOL[cfg.dtype]
    assert normwise_err(to_np(s_out[idx]), s_ref, dtype=cfg.dtype) <= TOL[cfg.dtype]
    nt.nt_device_status()


def test_block_one_long_sample(nt):
    """One 20,000-token sample beside three short ones (P = 400,000,010
    cells, a 102 GB bf16 pair state): element offsets far past 2^31, a pair
    row of 20,000 cells in the reduce, cell rows near the top of the 32-bit
    copy coordinates' range still far off.  Sampled cells (among them the
    first cells whose element offset passes 2^31 and 2^32) and rows against
    the oracle; the fused block's sampled cells bit for bit against the
    three calls', its m and s_out against the oracle."""
    lengths = [20000, 1, 0, 3]
    cfg = wl.PAIRFORMER_BF16
    torch.cuda.empty_cache()
    inp = wl.make_block_inputs(cfg, lengths=lengths, biases=True)
    part = nt.nt_partition_build(dev_lengths(inp.lengths))
    ref_part = opart.partition(inp.lengths)
    assert part.P == ref_part.P == 400_000_010
    w, ow = dev_weights(inp.blocks[0]), oracle_weights(inp.blocks[0])
    s = inp.s.to(DEV)
    z, m, s_out = nt.block_forward(part, s, w)
    rng = np.random.default_rng(2)
    edge = [(1 << 31) // cfg.C_z - 1, (1 << 31) // cfg.C_z, (1 << 32) // cfg.C_z]
    cells = np.concatenate([rng.integers(0, ref_part.P, size=500), ref_part.pair_off[1:-1] - 1,
                            ref_part.pair_off[:-1], [ref_part.P - 1], edge]).astype(np.int64)
    idx = torch.as_tensor(cells, device=DEV)
    got = z[idx].clone()
    _, Pt = oblock.block_cells(inp.lengths, f64(inp.s), ow, cells)
    assert normwise_err(to_np(got), Pt, dtype="bf16") <= TOL["bf16"]
    rows = np.array([0, 12345, 19999, 20000, 20001, 20003], dtype=np.int64)
    m_ref, s_ref = oblock.block_rows(inp.lengths, f64(inp.s), ow, rows)
    ridx = torch.as_tensor(rows, device=DEV)
    assert normwise_err(to_np(m[ridx]), m_ref, dtype="bf16") <= TOL["bf16"]
    assert normwise_err(to_np(s_out[ridx]), s_ref, dtype="bf16") <= TOL["bf16"]
    nt.nt_device_status()
    del z
    torch.cuda.empty_cache()
    zf, mf, sf = nt.nt_pair_block_fused(part, s, s, w)
    assert torch.equal(zf[idx], got)
    assert normwise_err(to_np(mf[ridx]), m_ref, dtype="bf16") <= TOL["bf16"]
    assert normwise_err(to_np(sf[ridx]), s_ref, dtype="bf16") <= TOL["bf16"]
    nt.nt_device_status()
    del zf
    torch.cuda.empty_cache()


def test_stacked_blocks_chain(nt):
    """Four blocks chained through the singles (the stacked workload's
    weights and width, lengths cut by 16): the library's chain against the
    oracle's own chain."""
    cfg = wl.STACKED4_BF16
    lengths = [n // 16 for n in cfg.fixed_lengths]
    inp = wl.make_block_inputs(cfg, lengths=lengths)
    part = nt.nt_partition_build(dev_lengths(inp.lengths))
    s = inp.s.to(DEV)
    for w in inp.blocks:
        z, m, s = nt.block_forward(part, s, dev_weights(w))
    x_ref, last = oblock.stacked_blocks(inp.lengths, f64(inp.s), [oracle_weights(w) for w in inp.blocks])
    assert normwise_err(to_np(s), x_ref, dtype="bf16") <= TOL["bf16"]
    assert normwise_err(to_np(z), last.z_tilde, dtype="bf16") <= TOL["bf16"]
    nt.nt_device_status()


# ----------------------------------------------------------------------------
# a5 varlen attention
# ----------------------------------------------------------------------------

def _attn_case(nt, seqlens, H, d, dtype, seed=0, lse=True):
    cfg = wl.AttnConfig("t", int(np.sum(seqlens)), 1, 1, H, d, dtype)
    a = wl.make_attn_inputs(cfg, seqlens=seqlens, seed=seed)
    cu = opart.partition(a.seqlens).cu_seqlens
    cu_d = torch.as_tensor(cu.astype(np.int32)).to(DEV)
    o, l = nt.nt_varlen_attn(a.q.to(DEV), a.k.to(DEV), a.v.to(DEV), cu_d, int(np.max(seqlens)),
                             want_lse=lse)
    return a, cu, o, l


@pytest.mark.parametrize("seqlens,H,d,dtype", [
    ([3, 1, 5, 0, 7, 64, 65, 130], 2, 64, "f32"),
    ([3, 1, 5, 0, 7, 64, 65, 130], 2, 64, "bf16"),
    ([200, 17, 1, 300, 129, 128, 127], 3, 64, "bf16"),
    ([40, 9, 77], 2, 32, "f32"),
    ([40, 9, 77], 2, 128, "bf16"),
    ([512], 12, 64, "bf16"),
    ([1000, 1537], 2, 64, "bf16"),          # mean length > 768: one CTA per (segment, tile, head)
    ([1, 2000, 3, 0, 5, 2, 1, 7, 9, 4000], 1, 64, "bf16"),   # mean 603: persistent, mostly empty tiles
])
def test_varlen_attention(nt, seqlens, H, d, dtype):
    a, cu, o, l = _attn_case(nt, seqlens, H, d, dtype)
    O_ref, lse_ref = oattn.varlen_attention(f64(a.q), f64(a.k), f64(a.v), cu)
    assert normwise_err(to_np(o), O_ref, dtype=dtype) <= TOL[dtype]
    assert np.abs(to_np(l) - lse_ref).max() <= (1e-4 if dtype == "f32" else 2e-2)
    nt.nt_device_status()


def test_varlen_attention_zero_leakage(nt):
    """Changing one segment's tokens leaves every other segment's output
    bit-identical ("Variable-length attention and data packing", failure
    mode: missing block-diagonal mask)."""
    seqlens = [37, 128, 5, 200, 64]
    a, cu, o, _ = _attn_case(nt, seqlens, 2, 64, "bf16")
    q, k, v = a.q.clone(), a.k.clone(), a.v.clone()
    lo, hi = int(cu[1]), int(cu[2])
    q[lo:hi] = -q[lo:hi]
    k[lo:hi] = k[lo:hi] * 3
    v[lo:hi] = 7.0
    cu_d = torch.as_tensor(cu.astype(np.int32)).to(DEV)
    o2, _ = nt.nt_varlen_attn(q.to(DEV), k.to(DEV), v.to(DEV), cu_d, 200)
    assert torch.equal(o2[:lo], o[:lo]) and torch.equal(o2[hi:], o[hi:])
    # a constant V comes back as that constant, within the bf16 tolerance: the
    # kernel normalises by a running max that may trail the true one, so the
    # largest probability is not exactly 1 and P's bf16 rounding stays visible
    assert normwise_err(to_np(o2[lo:hi]), np.full((hi - lo, 2, 64), 7.0), dtype="bf16") <= TOL["bf16"]


def test_varlen_attention_full_size_sampled(nt):
    """The packed stream of 65,536 tokens, 237 segments, 12 heads x 64:
    every output of a sample of segments (first, last, longest, shortest
    and random ones) against the oracle."""
    cfg = wl.VARLEN_ATTN_BF16
    a = wl.make_attn_inputs(cfg)
    cu = opart.partition(a.seqlens).cu_seqlens
    cu_d = torch.as_tensor(cu.astype(np.int32)).to(DEV)
    o, l = nt.nt_varlen_attn(a.q.to(DEV), a.k.to(DEV), a.v.to(DEV), cu_d, int(a.seqlens.max()),
                             want_lse=True)
    B = len(a.seqlens)
    segs = sorted(set([0, B - 1, int(np.argmax(a.seqlens)), int(np.argmin(a.seqlens))] +
                      list(np.random.default_rng(2).integers(0, B, size=8))))
    O_ref, lse_ref = oattn.varlen_attention(f64(a.q), f64(a.k), f64(a.v), cu, segments=segs)
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in segs])
    idx = torch.as_tensor(rows, device=DEV)
    assert normwise_err(to_np(o[idx]), O_ref[rows], dtype="bf16") <= TOL["bf16"]
    assert np.abs(to_np(l[:, idx]) - lse_ref[:, rows]).max() <= 2e-2
    nt.nt_device_status()


def test_varlen_attention_bad_cu_flagged(nt):
    """cu_seqlens whose last entry exceeds T is caught by the kernel's own
    bounds check (status word), with no access beyond the buffers."""
    T, H, d = 64, 1, 64
    q = torch.zeros(T, H, d, dtype=torch.bfloat16, device=DEV)
    cu_bad = torch.tensor([0, 32, 96], dtype=torch.int32, device=DEV)
    nt.nt_varlen_attn(q, q, q, cu_bad, 64)
    with pytest.raises(nt.NTError) as ei:
        nt.nt_device_status()
    assert ei.value.status == 6
    # the same check on the one-CTA-per-item schedule (mean length > 768)
    T = 2048
    q = torch.zeros(T, H, d, dtype=torch.bfloat16, device=DEV)
    cu_bad = torch.tensor([0, 1000, 2500], dtype=torch.int32, device=DEV)
    nt.nt_varlen_attn(q, q, q, cu_bad, 1500)
    with pytest.raises(nt.NTError) as ei:
        nt.nt_device_status()
    assert ei.value.status == 6
