"""GPU parity of the torch.autograd bindings (variable_length_batching_gb300
.autograd): the Eq. 5 loss written in plain torch ops on pair_block's
outputs ("DanLing NestedTensor" Appendix A.1), back-propagated through the
Function, gives the oracle's gradients; varlen_attention's gradients equal
nt_varlen_attn_bwd's bit for bit and a per-segment fp32 softmax attention's
within tolerance."""
import math

import numpy as np
import pytest
import torch

from _helpers import TOL, f64, normwise_err, oracle_weights, to_np
from oracle import block as oblock
from oracle import block_backward as obwd
from variable_length_batching_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_batching_gb300 import autograd, build, nt as ntmod
    build.build()
    return ntmod, autograd


def _eq5_torch(lengths, s_out, z_t):
    """Eq. 5 in torch ops (fp32), S = 1, square pairs."""
    B = len(lengths)
    T = int(sum(lengths))
    P = int(sum(n * n for n in lengths))
    C, Cp = s_out.shape[1], z_t.shape[1]
    lx = s_out.new_zeros((), dtype=torch.float32)
    lp = s_out.new_zeros((), dtype=torch.float32)
    r = c = 0
    for i, n in enumerate(lengths):
        a, b = 1.0 + i / B, 1.5 - i / (2.0 * B)
        x = s_out[r:r + n].float()
        p = z_t[c:c + n * n].float()
        lx = lx + a * (x * x).sum()
        lp = lp + b * (p * p).sum()
        r += n
        c += n * n
    return lx / (C * T) + lp / (Cp * P)


@pytest.mark.parametrize("cfg,lengths,biases", [(wl.TINY_FP32, [5, 0, 9, 1], True),
                                                (wl.PAIRFORMER_BF16, [37, 1, 0, 70], True)])
def test_pair_block_autograd(mods, cfg, lengths, biases):
    nt, ag = mods
    inp = wl.make_block_inputs(cfg, lengths=lengths, biases=biases)
    w = inp.blocks[0]
    leaf = lambda t: None if t is None else t.to(DEV).clone().requires_grad_(True)
    s = leaf(inp.s)
    params = [leaf(t) for t in (w.W_a, w.W_b, w.ln_gamma, w.ln_beta, w.W1, w.b1, w.W2, w.b2, w.W_g, w.b_g)]
    part = nt.nt_partition_build(torch.as_tensor(np.asarray(inp.lengths, dtype=np.int32)).to(DEV))
    z_t, s_out = ag.pair_block(part, s, *params)
    loss = _eq5_torch(list(inp.lengths), s_out, z_t)
    loss.backward()
    torch.cuda.synchronize()
    nt.nt_device_status()
    ow = oracle_weights(w)
    fwd = oblock.block_packed(inp.lengths, f64(inp.s), ow)
    ref_loss, ref = obwd.block_loss_and_grads(inp.lengths, f64(inp.s), ow, fwd.z_tilde, fwd.s_out)
    assert abs(float(loss.detach()) - ref_loss) <= (1e-5 if cfg.dtype == "f32" else 2e-2) * abs(ref_loss)
    names = ("ds", "dW_a", "dW_b", "dgamma", "dbeta", "dW1", "db1", "dW2", "db2", "dW_g", "db_g")
    for name, t in zip(names, [s] + params):
        assert t.grad is not None and t.grad.dtype == t.dtype, name
        e = normwise_err(to_np(t.grad), getattr(ref, name), dtype=cfg.dtype)
        assert e <= TOL[cfg.dtype], f"{name}: {e:.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_attention_autograd(mods, causal):
    nt, ag = mods
    seqlens = [5, 130, 1, 64, 200]
    H, d = 2, 64
    T = sum(seqlens)
    g = torch.Generator(device=DEV).manual_seed(3)
    mk = lambda: torch.randn(T, H, d, device=DEV, generator=g).to(torch.bfloat16)
    q, k, v = mk(), mk(), mk()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32), device=DEV)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = ag.varlen_attention(qa, ka, va, cu, max(seqlens), causal=causal)
    d_o = torch.randn(T, H, d, device=DEV, generator=g).to(torch.bfloat16)
    o.backward(d_o)
    torch.cuda.synchronize()
    nt.nt_device_status()
    # the same as the direct calls, bit for bit
    o2, lse = nt.nt_varlen_attn_qk(q, k, v, cu, cu, max(seqlens), causal=causal, want_lse=True)
    dq, dk, dv = nt.nt_varlen_attn_bwd(q, k, v, o2, d_o, lse, cu, None, max(seqlens), causal=causal)
    assert torch.equal(o, o2)
    assert torch.equal(qa.grad, dq) and torch.equal(ka.grad, dk) and torch.equal(va.grad, dv)
    # and a per-segment fp32 softmax attention's gradients
    qf, kf, vf = (t.float().clone().requires_grad_(True) for t in (q, k, v))
    outs = []
    r = 0
    for n in seqlens:
        s_ = torch.einsum("qhd,khd->hqk", qf[r:r + n], kf[r:r + n]) / math.sqrt(d)
        if causal:
            s_ = s_.masked_fill(torch.ones(n, n, device=DEV, dtype=torch.bool).triu(1), float("-inf"))
        outs.append(torch.einsum("hqk,khd->qhd", torch.softmax(s_, -1), vf[r:r + n]))
        r += n
    torch.cat(outs).backward(d_o.float())
    for got, want in ((qa.grad, qf.grad), (ka.grad, kf.grad), (va.grad, vf.grad)):
        assert normwise_err(to_np(got), to_np(want), dtype="bf16") <= TOL["bf16"]
