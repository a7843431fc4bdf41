"""GPU parity of the fused block (nt_pair_block_fused): the single -> pair ->
single block of "DanLing NestedTensor" Eq. 1 in one pass over the pair
state.  Its z~ must equal the three separate calls' bit for bit (same
roundings); m and s_out must match the oracle within the bf16/fp32
tolerances (only the order of the fp32 row sums differs)."""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

from _helpers import TOL, f64, normwise_err, oracle_weights, to_np
from oracle import block as oblock
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


def _dw(w):
    g = lambda t: None if t is None else t.to(DEV).contiguous()
    return SimpleNamespace(W_a=g(w.W_a), W_b=g(w.W_b), ln_gamma=g(w.ln_gamma), ln_beta=g(w.ln_beta),
                           W1=g(w.W1), b1=g(w.b1), W2=g(w.W2), b2=g(w.b2), W_g=g(w.W_g), b_g=g(w.b_g))


def _dev(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).to(DEV)


@pytest.mark.parametrize("cfg,lengths,biases", [
    (wl.PAIRFORMER_BF16, None, False),
    (wl.PAIRFORMER_BF16, [0, 1, 7, 0, 130, 2, 1, 33], True),
    (wl.LOGNORMAL_BF16, None, True),
    (wl.TINY_FP32, None, True),                     # not fusable: the three calls' kernels
])
def test_fused_block_square(nt, cfg, lengths, biases):
    inp = wl.make_block_inputs(cfg, lengths=lengths, biases=biases)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build(_dev(inp.lengths))
    s = inp.s.to(DEV)
    zf, mf, sf = nt.nt_pair_block_fused(part, s, s, w)
    zu, mu, su = nt.block_forward(part, s, w)
    assert torch.equal(zf, zu)                      # same roundings, same kernels for z~
    tol = TOL[cfg.dtype]
    assert normwise_err(to_np(mf), to_np(mu), dtype=cfg.dtype) <= tol and normwise_err(to_np(sf), to_np(su), dtype=cfg.dtype) <= tol
    if cfg.name != wl.LOGNORMAL_BF16.name:          # the dense oracle on the small batches
        ref = oblock.block_packed(inp.lengths, f64(inp.s), oracle_weights(inp.blocks[0]))
        assert normwise_err(to_np(zf), ref.z_tilde, dtype=cfg.dtype) <= tol
        assert normwise_err(to_np(mf), ref.m, dtype=cfg.dtype) <= tol
        assert normwise_err(to_np(sf), ref.s_out, dtype=cfg.dtype) <= tol
    nt.nt_device_status()


@pytest.mark.parametrize("rows,cols", [(None, None), ([0, 3, 130, 1, 64, 2, 0, 9], [5, 0, 7, 200, 1, 64, 3, 128])])
def test_fused_block_rect(nt, rows, cols):
    cfg = wl.RECT_BF16
    inp = wl.make_rect_inputs(cfg, rows=rows, cols=cols, biases=True)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build_rect(_dev(inp.rows), _dev(inp.cols))
    sr, sc = inp.s_row.to(DEV), inp.s_col.to(DEV)
    zf, mf, sf = nt.nt_pair_block_fused(part, sr, sc, w)
    ref = oblock.block_packed_rect(inp.rows, inp.cols, f64(inp.s_row), f64(inp.s_col), oracle_weights(inp.blocks[0]))
    zu, mu, su = nt.block_forward(part, sr, w, s_col=sc)
    assert torch.equal(zf, zu)
    assert normwise_err(to_np(zf), ref.z_tilde, dtype="bf16") <= TOL["bf16"]
    assert normwise_err(to_np(mf), ref.m, dtype="bf16") <= TOL["bf16"]
    assert normwise_err(to_np(sf), ref.s_out, dtype="bf16") <= TOL["bf16"]
    nt.nt_device_status()


def test_fused_block_swiglu(nt):
    cfg = wl.PAIRFORMER_BF16
    inp = wl.make_block_inputs(cfg, lengths=[64, 1, 200, 0, 37, 5, 128, 90])
    w = _dw(inp.blocks[0])
    sw = wl.make_swiglu_weights(cfg.C_z, cfg.H_t, "bf16", biases=True, seed=3)
    w.W1, w.b1, w.W2, w.b2 = sw.W1.to(DEV), sw.b1.to(DEV), sw.W2.to(DEV), sw.b2.to(DEV)
    W3, b3 = sw.W3.to(DEV), sw.b3.to(DEV)
    part = nt.nt_partition_build(_dev(inp.lengths))
    s = inp.s.to(DEV)
    zf, mf, sf = nt.nt_pair_block_fused(part, s, s, w, W3=W3, b3=b3)
    z = nt.nt_pair_broadcast(part, s, s, w.W_a, w.W_b)
    zu = nt.nt_pair_transition_swiglu(part, z, w.ln_gamma, w.ln_beta, w.W1, w.b1, W3, b3, w.W2, w.b2)
    mu, su = nt.nt_pair_reduce(part, zu, w.W_g, w.b_g, s_in=s)
    assert torch.equal(zf, zu)
    assert normwise_err(to_np(mf), to_np(mu), dtype="bf16") <= TOL["bf16"]
    assert normwise_err(to_np(sf), to_np(su), dtype="bf16") <= TOL["bf16"]
    nt.nt_device_status()


def test_fused_block_twice_in_a_row(nt):
    """The row-sum accumulator is cleared on every call: two calls agree."""
    inp = wl.make_block_inputs(wl.PAIRFORMER_BF16)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build(_dev(inp.lengths))
    s = inp.s.to(DEV)
    ws = torch.empty(nt.lib().nt_pair_block_fused_workspace_bytes(part.T, part.T_cols, 128), dtype=torch.uint8,
                     device=DEV)
    z1, m1, s1 = nt.nt_pair_block_fused(part, s, s, w, workspace=ws)
    m1, s1 = m1.clone(), s1.clone()
    z2, m2, s2 = nt.nt_pair_block_fused(part, s, s, w, workspace=ws)
    assert torch.equal(z1, z2)
    assert normwise_err(to_np(m2), to_np(m1)) <= 1e-3 and normwise_err(to_np(s2), to_np(s1)) <= 1e-3
