"""GPU parity of the Eq. 5 loss and of the block's backward
("DanLing NestedTensor" Appendix A.1, Eq. 5; the chain rule of Eq. 1)
against the CPU oracle on the same seeded inputs: the loss within 1e-5
relative (fp32 accumulation of the squared sums), every gradient normwise
within 2e-2 (bf16 I/O) or 1e-5 (fp32), the oracle running its own forward
on the exact inputs."""
import numpy as np
import pytest
import torch

from _helpers import TOL, f64, normwise_err, oracle_weights, to_np
from oracle import block as oblock
from oracle import block_backward as obwd
from variable_length_batching_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
NAMES = ("ds", "dW_a", "dW_b", "dgamma", "dbeta", "dW1", "db1", "dW2", "db2", "dW_g", "db_g")


@pytest.fixture(scope="module")
def nt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_batching_gb300 import build, nt as ntmod
    build.build()
    return ntmod


def _dw(w):
    from types import SimpleNamespace
    d = lambda t: None if t is None else t.to(DEV)
    return SimpleNamespace(W_a=d(w.W_a), W_b=d(w.W_b), ln_gamma=d(w.ln_gamma), ln_beta=d(w.ln_beta), W1=d(w.W1),
                           b1=d(w.b1), W2=d(w.W2), b2=d(w.b2), W_g=d(w.W_g), b_g=d(w.b_g))


def _run(nt, cfg, lengths, biases, seed=0):
    inp = wl.make_block_inputs(cfg, lengths=lengths, biases=biases, seed=seed)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build(torch.as_tensor(inp.lengths).to(DEV))
    s = inp.s.to(DEV)
    z, m, s_out = nt.block_forward(part, s, w)
    loss, ds_out, dz = nt.nt_pair_block_loss(part, s_out, z)
    g = nt.nt_pair_block_backward(part, s, w, m, ds_out, dz)
    torch.cuda.synchronize()
    nt.nt_device_status()
    ow = oracle_weights(inp.blocks[0])
    fwd = oblock.block_packed(inp.lengths, f64(inp.s), ow)
    ref_loss, ref = obwd.block_loss_and_grads(inp.lengths, f64(inp.s), ow, fwd.z_tilde, fwd.s_out)
    return float(loss.item()), g, ref_loss, ref, cfg.dtype


def _check(loss, g, ref_loss, ref, dtype, names=NAMES):
    assert abs(loss - ref_loss) <= (1e-5 if dtype == "f32" else 2e-2) * abs(ref_loss)
    for n in names:
        got, want = to_np(g[n]), getattr(ref, n)
        assert got.shape == want.shape, n
        e = normwise_err(got, want, dtype=dtype)
        assert e <= TOL[dtype], f"{n}: normwise error {e:.3e}"


@pytest.mark.parametrize("lengths,biases", [(None, True), ([3, 0, 1, 17], False), ([1], True)])
def test_block_backward_tiny_fp32(nt, lengths, biases):
    _check(*_run(nt, wl.TINY_FP32, lengths, biases))


@pytest.mark.parametrize("lengths,biases", [([37, 1, 0, 70], True), ([64, 31, 5], False)])
def test_block_backward_bf16(nt, lengths, biases):
    _check(*_run(nt, wl.PAIRFORMER_BF16, lengths, biases))


def test_block_backward_bf16_cuda_core_route(nt):
    """bf16 at C_z = 64 (not the tensor-core route's 128): the CUDA-core
    kernels, against the oracle."""
    _check(*_run(nt, _cz64(), [40, 3, 0, 25], True))


def test_tensor_core_weight_gradients_reproducible(nt):
    """dW1, db1, dW2 and db2 of the tensor-core route are summed over fixed
    cell splits in a fixed order, and du, dv (hence ds) over fixed 32 x 32
    cell items: two calls give the same bits."""
    inp = wl.make_block_inputs(wl.PAIRFORMER_BF16)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build(torch.as_tensor(inp.lengths).to(DEV))
    s = inp.s.to(DEV)
    z, m, s_out = nt.block_forward(part, s, w)
    _, ds_out, dz = nt.nt_pair_block_loss(part, s_out, z)
    g1 = nt.nt_pair_block_backward(part, s, w, m, ds_out, dz)
    g2 = nt.nt_pair_block_backward(part, s, w, m, ds_out, dz)
    torch.cuda.synchronize()
    for n in ("ds", "dW1", "db1", "dW2", "db2"):
        assert torch.equal(g1[n], g2[n]), n


def _cz64():
    import dataclasses
    return dataclasses.replace(wl.PAIRFORMER_BF16, name="bf16_Cz64", C_s=128, C_z=64, H_t=256)


@pytest.mark.parametrize("route", ["tensor_core", "tensor_core_batch", "cuda_core_f32", "cuda_core_bf16"])
def test_loss_backward_equals_two_calls(nt, route):
    """nt_pair_block_loss_backward against nt_pair_block_loss followed by
    nt_pair_block_backward on the same inputs: the same loss bits on every
    route; on the tensor-core route (where dL/dz~ = gp_i z~ is formed from
    z~ where it is read) also the same ds and split-summed weight gradients,
    bit for bit.  The gradients accumulated with fp32 atomics differ between
    any two calls by the order of their sums: within 1e-5 normwise (one
    reordering of an fp32 sum of a few thousand terms, with some
    cancellation; two plain calls were seen 1.0e-6 apart on dbeta)."""
    cfg, lengths = {"tensor_core": (wl.PAIRFORMER_BF16, [33, 0, 1, 32, 31, 65, 37]),
                    "tensor_core_batch": (wl.PAIRFORMER_BF16, None),
                    "cuda_core_f32": (wl.TINY_FP32, [5, 0, 9, 1]),
                    "cuda_core_bf16": (_cz64(), [40, 3, 0, 25])}[route]
    inp = wl.make_block_inputs(cfg, lengths=lengths, biases=True, seed=4)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build(torch.as_tensor(inp.lengths).to(DEV))
    s = inp.s.to(DEV)
    z, m, s_out = nt.block_forward(part, s, w)
    l1, ds_out, dz = nt.nt_pair_block_loss(part, s_out, z)
    g1 = nt.nt_pair_block_backward(part, s, w, m, ds_out, dz)
    l2, g2 = nt.nt_pair_block_loss_backward(part, s, w, m, s_out, z)
    torch.cuda.synchronize()
    nt.nt_device_status()
    assert torch.equal(l1, l2)
    exact = ("ds", "dW1", "db1", "dW2", "db2") if route.startswith("tensor_core") else ()
    for n in NAMES:
        if n in exact:
            assert torch.equal(g1[n], g2[n]), n
        else:
            assert normwise_err(to_np(g2[n]), to_np(g1[n]), dtype="f32") <= 1e-5, n


def test_loss_backward_against_oracle(nt):
    """The fused call on a bf16 batch with 31-, 32- and 33-token samples (the
    edges of the 32 x 32 cell items), against the oracle."""
    inp = wl.make_block_inputs(wl.PAIRFORMER_BF16, lengths=[33, 0, 1, 32, 31, 65], biases=True, seed=6)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build(torch.as_tensor(inp.lengths).to(DEV))
    s = inp.s.to(DEV)
    z, m, s_out = nt.block_forward(part, s, w)
    loss, g = nt.nt_pair_block_loss_backward(part, s, w, m, s_out, z)
    torch.cuda.synchronize()
    nt.nt_device_status()
    ow = oracle_weights(inp.blocks[0])
    fwd = oblock.block_packed(inp.lengths, f64(inp.s), ow)
    ref_loss, ref = obwd.block_loss_and_grads(inp.lengths, f64(inp.s), ow, fwd.z_tilde, fwd.s_out)
    _check(float(loss.item()), g, ref_loss, ref, "bf16")


def test_block_backward_pairformer_batch(nt):
    """The B=8 Pairformer-style batch itself (N_i ~ U[64, 256], P = 157,023)."""
    _check(*_run(nt, wl.PAIRFORMER_BF16, None, False))


def test_loss_is_reproducible(nt):
    """The loss sums its partials in a fixed order: two calls give the same bits."""
    inp = wl.make_block_inputs(wl.PAIRFORMER_BF16)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build(torch.as_tensor(inp.lengths).to(DEV))
    z, m, s_out = nt.block_forward(part, inp.s.to(DEV), w)
    l1, _, _ = nt.nt_pair_block_loss(part, s_out, z, want_grads=False)
    l2, _, _ = nt.nt_pair_block_loss(part, s_out, z, want_grads=False)
    torch.cuda.synchronize()
    assert torch.equal(l1, l2)


def test_rectangular_partition_refused(nt):
    part = nt.nt_partition_build_rect(torch.tensor([3, 2], dtype=torch.int32, device=DEV),
                                      torch.tensor([4, 1], dtype=torch.int32, device=DEV))
    inp = wl.make_block_inputs(wl.TINY_FP32, lengths=[3, 2])
    w = _dw(inp.blocks[0])
    s = inp.s.to(DEV)
    ds_out = torch.zeros(5, s.shape[1], device=DEV)
    m = torch.zeros(5, 16, device=DEV)
    with pytest.raises(nt.NTError) as e:
        nt.nt_pair_block_backward(part, s, w, m, ds_out)
    assert e.value.status == 2


def test_block_backward_near_uniform_sampled(nt):
    """The near-uniform B=16 batch itself (P = 8.6 M cells, the size the bench
    times): the loss and backward of the whole batch on the GPU, through the
    one-call entry and through the two calls (the same loss and ds bits), and
    the single-row gradient ds of its shortest sample against the oracle, which
    needs that sample alone (ds of a sample's rows depends on its own cells;
    Eq. 5's weights and totals are the batch's)."""
    cfg = wl.NEAR_UNIFORM_BF16
    inp = wl.make_block_inputs(cfg)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build(torch.as_tensor(inp.lengths).to(DEV))
    s = inp.s.to(DEV)
    z, m, s_out = nt.block_forward(part, s, w)
    # the one-call entry the bench times, then the two calls it must equal
    l1, g1 = nt.nt_pair_block_loss_backward(part, s, w, m, s_out, z)
    l2, ds_out, dz = nt.nt_pair_block_loss(part, s_out, z)
    del z
    g = nt.nt_pair_block_backward(part, s, w, m, ds_out, dz)
    torch.cuda.synchronize()
    nt.nt_device_status()
    assert torch.equal(l1, l2)
    assert torch.equal(g1["ds"], g["ds"])
    lengths = np.asarray(inp.lengths, dtype=np.int64)
    k = int(np.argmin(lengths))
    n = int(lengths[k])
    r0 = int(lengths[:k].sum())
    B, T, P = len(lengths), int(lengths.sum()), int((lengths ** 2).sum())
    ow = oracle_weights(inp.blocks[0])
    X = f64(inp.s)[r0:r0 + n]
    res = oblock.block_sample(X, ow)
    alpha, beta = obwd.eq5_sample_weights(B)
    C, Cp = X.shape[1], res.P_tilde.shape[2]
    dX_up = 2.0 * alpha[k] * res.X_tilde / (C * T)
    dP_up = 2.0 * beta[k] * res.P_tilde / (Cp * P)
    ref_ds, _ = obwd.block_backward_sample(X, ow, dX_up, dP_up)
    got = to_np(g1["ds"][r0:r0 + n])
    e = normwise_err(got, ref_ds, dtype="bf16")
    assert e <= TOL["bf16"], f"ds of sample {k} (N = {n}): {e:.3e}"


@pytest.mark.parametrize("cfg", [wl.TINY_FP32, wl.PAIRFORMER_BF16])
def test_empty_batch(nt, cfg):
    """Samples that all have length 0 (T = P = 0): the forward calls, the
    fused block, the loss and the backward through both entries accept the
    empty tensors; Eq. 5's empty sums give a loss of 0 (the oracle's
    reading), every parameter gradient is 0 and ds is empty."""
    inp = wl.make_block_inputs(cfg, lengths=[0, 0], biases=True)
    w = _dw(inp.blocks[0])
    part = nt.nt_partition_build(torch.as_tensor(np.asarray(inp.lengths, dtype=np.int32)).to(DEV))
    assert (part.T, part.P) == (0, 0)
    s = inp.s.to(DEV)
    assert s.shape[0] == 0
    z, m, s_out = nt.block_forward(part, s, w)
    assert z.shape == (0, cfg.C_z) and m.shape == (0, cfg.C_z) and s_out.shape == (0, cfg.C_s)
    zf, mf, sf = nt.nt_pair_block_fused(part, s, s, w)
    assert zf.shape == (0, cfg.C_z) and sf.shape == (0, cfg.C_s)
    loss, ds_out, dz = nt.nt_pair_block_loss(part, s_out, z)
    g = nt.nt_pair_block_backward(part, s, w, m, ds_out, dz)
    l1, g1 = nt.nt_pair_block_loss_backward(part, s, w, m, s_out, z)
    torch.cuda.synchronize()
    assert nt.nt_device_status() == 0
    ref_loss = obwd.eq5_loss(inp.lengths, np.zeros((0, cfg.C_s)), np.zeros((0, cfg.C_z)))
    assert ref_loss == 0.0
    assert float(loss.item()) == 0.0 and float(l1.item()) == 0.0
    for grads in (g, g1):
        assert grads["ds"].shape == (0, cfg.C_s)
        for n in NAMES[1:]:
            assert torch.count_nonzero(grads[n]).item() == 0, n
