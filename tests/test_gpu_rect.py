"""GPU parity of rectangular pair states ("DanLing NestedTensor" section 3.2
"Consuming one logical axis", Eq. 4; Appendix A.1, rectangular variant):
N_i x M_i cells with distinct row and column singles, column mean divided by
M_i.  Partitions bit-exact; floats normwise against the CPU oracle
(2e-2 bf16, 1e-5 fp32)."""
import numpy as np
import pytest
import torch

from _helpers import TOL, f64, normwise_err, oracle_weights, to_np
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


def _dev(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).to(DEV)


def _dev_weights(w):
    from types import SimpleNamespace
    g = lambda t: None if t is None else t.to(DEV).contiguous()
    return SimpleNamespace(W_a=g(w.W_a), W_b=g(w.W_b), ln_gamma=g(w.ln_gamma), ln_beta=g(w.ln_beta),
                           W1=g(w.W1), b1=g(w.b1), W2=g(w.W2), b2=g(w.b2), W_g=g(w.W_g), b_g=g(w.b_g))


_r = np.random.default_rng(5)
RECT_PARTITIONS = [
    ([2, 3], [4, 1]),
    ([0, 3, 2], [2, 0, 5]),
    ([1] * 33, list(range(33))),
    ([], []),
    (list(_r.integers(0, 40, 1500)), list(_r.integers(0, 40, 1500))),   # B > 1024: carries across chunks
    (list(wl.make_rect_inputs(wl.RECT_BF16).rows), list(wl.make_rect_inputs(wl.RECT_BF16).cols)),
]


@pytest.mark.parametrize("rows,cols", RECT_PARTITIONS)
def test_rect_partition_bit_exact(nt, rows, cols):
    part = nt.nt_partition_build_rect(_dev(rows), _dev(cols))
    ref = opart.partition_rect(rows, cols)
    assert (part.T, part.T_cols, part.P, part.max_len, part.max_col_len) == \
        (ref.T_rows, ref.T_cols, ref.P, ref.max_rows, ref.max_cols)
    assert np.array_equal(part.cu_seqlens.cpu().numpy(), ref.cu_rows)
    assert np.array_equal(part.col_cu_seqlens.cpu().numpy(), ref.cu_cols)
    assert np.array_equal(part.pair_off.cpu().numpy(), ref.pair_off)
    assert np.array_equal(part.row_start.cpu().numpy(), ref.row_start)
    if ref.T_rows:
        assert np.array_equal(part.row_sample[:ref.T_rows].cpu().numpy(), ref.row_sample)


@pytest.mark.parametrize("cfg,rows,cols,biases", [
    (wl.RECT_TINY_FP32, None, None, False),
    (wl.RECT_TINY_FP32, [3, 0, 5, 2], [0, 4, 1, 6], True),        # M_i = 0 rows, N_i = 0 columns
    (wl.RECT_BF16, None, None, False),
    (wl.RECT_BF16, [0, 3, 130, 1, 64, 2, 0, 9], [5, 0, 7, 200, 1, 64, 3, 128], True),
])
def test_rect_block(nt, cfg, rows, cols, biases):
    inp = wl.make_rect_inputs(cfg, rows=rows, cols=cols, biases=biases)
    w = inp.blocks[0]
    part = nt.nt_partition_build_rect(_dev(inp.rows), _dev(inp.cols))
    z, m, s_out = nt.block_forward(part, inp.s_row.to(DEV), _dev_weights(w), s_col=inp.s_col.to(DEV))
    ref = oblock.block_packed_rect(inp.rows, inp.cols, f64(inp.s_row), f64(inp.s_col), oracle_weights(w))
    tol = TOL[cfg.dtype]
    assert z.shape == (ref.z_tilde.shape[0], cfg.C_z)
    assert normwise_err(to_np(z), ref.z_tilde, dtype=cfg.dtype) <= tol
    assert normwise_err(to_np(m), ref.m, dtype=cfg.dtype) <= tol
    assert normwise_err(to_np(s_out), ref.s_out, dtype=cfg.dtype) <= tol
    # rows of a sample with M_i = 0 have exact zero means
    cu = np.concatenate([[0], np.cumsum(inp.rows)])
    for i in np.nonzero(np.asarray(inp.cols) == 0)[0]:
        assert torch.count_nonzero(m[cu[i]:cu[i + 1]]).item() == 0
    nt.nt_device_status()


def test_rect_broadcast_alone(nt):
    """The broadcast before the transition, cell by cell against the oracle."""
    cfg = wl.RECT_BF16
    inp = wl.make_rect_inputs(cfg)
    w = inp.blocks[0]
    part = nt.nt_partition_build_rect(_dev(inp.rows), _dev(inp.cols))
    z = nt.nt_pair_broadcast(part, inp.s_row.to(DEV), inp.s_col.to(DEV), w.W_a.to(DEV), w.W_b.to(DEV))
    ref = oblock.pair_broadcast_rect(inp.rows, inp.cols, f64(inp.s_row), f64(inp.s_col), f64(w.W_a), f64(w.W_b))
    assert normwise_err(to_np(z), ref, dtype="bf16") <= TOL["bf16"]


def test_rect_with_equal_lengths_is_the_square_path(nt):
    """nt_partition_build_rect(N, N) gives the square partition, and the block
    on it is bit-identical to the block on the square partition."""
    cfg = wl.PAIRFORMER_BF16
    inp = wl.make_block_inputs(cfg, lengths=[37, 0, 128, 5, 64, 1, 200, 9])
    ps = nt.nt_partition_build(_dev(inp.lengths))
    pr = nt.nt_partition_build_rect(_dev(inp.lengths), _dev(inp.lengths))
    for a, b in ((ps.cu_seqlens, pr.cu_seqlens), (ps.cu_seqlens, pr.col_cu_seqlens), (ps.pair_off, pr.pair_off),
                 (ps.row_start, pr.row_start)):
        assert torch.equal(a, b)
    w = _dev_weights(inp.blocks[0])
    s = inp.s.to(DEV)
    z1, m1, s1 = nt.block_forward(ps, s, w)
    z2, m2, s2 = nt.block_forward(pr, s, w, s_col=s)
    assert torch.equal(z1, z2) and torch.equal(m1, m2) and torch.equal(s1, s2)


def test_rect_column_leakage(nt):
    """Changing one sample's column singles changes only that sample's cells."""
    cfg = wl.RECT_TINY_FP32
    inp = wl.make_rect_inputs(cfg, rows=[4, 6, 3], cols=[5, 2, 7])
    w = _dev_weights(inp.blocks[0])
    part = nt.nt_partition_build_rect(_dev(inp.rows), _dev(inp.cols))
    sr, sc = inp.s_row.to(DEV), inp.s_col.to(DEV)
    z1 = nt.nt_pair_broadcast(part, sr, sc, w.W_a, w.W_b)
    sc2 = sc.clone()
    sc2[5:7] += 3.0                                    # sample 1's two column singles
    z2 = nt.nt_pair_broadcast(part, sr, sc2, w.W_a, w.W_b)
    po = opart.partition_rect(inp.rows, inp.cols).pair_off
    assert torch.equal(z1[:po[1]], z2[:po[1]]) and torch.equal(z1[po[2]:], z2[po[2]:])
    assert not torch.equal(z1[po[1]:po[2]], z2[po[1]:po[2]])


def test_rect_noalloc_matches_workspace_call(nt):
    """The allocation-free broadcast handles rectangular partitions, with the
    same result as the call given a workspace."""
    inp = wl.make_rect_inputs(wl.RECT_BF16)
    w = _dev_weights(inp.blocks[0])
    part = nt.nt_partition_build_rect(_dev(inp.rows), _dev(inp.cols))
    sr, sc = inp.s_row.to(DEV), inp.s_col.to(DEV)
    z1 = nt.nt_pair_broadcast(part, sr, sc, w.W_a, w.W_b)
    z2 = nt.nt_pair_broadcast_noalloc(part, sr, sc, w.W_a, w.W_b)
    assert torch.equal(z1, z2)
