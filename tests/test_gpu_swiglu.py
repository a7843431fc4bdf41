"""GPU parity of the SwiGLU transition ("DanLing NestedTensor" Eq. 1: h is a
SwiGLU feature update): z~ = z + W2 (SiLU(W1 LN(z) + b1) * (W3 LN(z) + b3)) + b2
against the CPU oracle on the same seeded inputs, normwise (2e-2 bf16,
1e-5 fp32)."""
import numpy as np
import pytest
import torch

from _helpers import TOL, f64, normwise_err, to_np
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


def _run(nt, lengths, C_z, H_t, dtype, biases, seed=0, in_place=False):
    part = nt.nt_partition_build(torch.as_tensor(np.asarray(lengths, dtype=np.int32)).to(DEV))
    P = opart.partition(lengths).P
    z = wl.random_rows(P, C_z, dtype, seed=seed + 11, scale=1.5)
    w = wl.make_swiglu_weights(C_z, H_t, dtype, biases=biases, seed=seed)
    d = lambda t: None if t is None else t.to(DEV)
    zd = z.to(DEV)
    out = nt.nt_pair_transition_swiglu(part, zd, d(w.ln_gamma), d(w.ln_beta), d(w.W1), d(w.b1), d(w.W3), d(w.b3),
                                       d(w.W2), d(w.b2), out=zd if in_place else None)
    return z, w, out


def _ref(z, w, rows=None):
    zz = f64(z) if rows is None else f64(z)[rows]
    g = lambda t: None if t is None else f64(t)
    return oblock.transition_swiglu(zz, g(w.ln_gamma), g(w.ln_beta), 1e-5, g(w.W1), g(w.b1), g(w.W3), g(w.b3),
                                    g(w.W2), g(w.b2))


@pytest.mark.parametrize("lengths,C_z,H_t,dtype,biases,in_place", [
    ([64, 1, 200, 0, 37], 128, 512, "bf16", False, False),   # tensor cores, 8 chunks of 64
    ([64, 1, 200, 0, 37], 128, 512, "bf16", True, True),     # biases, in place
    ([31, 17, 90], 128, 192, "bf16", True, False),           # 3 chunks: odd chunk count
    ([31, 17, 90], 128, 64, "bf16", False, False),           # one chunk
    ([9, 20, 4], 64, 256, "bf16", True, False),              # CUDA cores (C_z != 128)
    ([9, 20, 4], 16, 64, "f32", True, False),                # fp32 mode
    ([9, 20, 4], 128, 512, "f32", False, False),
])
def test_swiglu_transition(nt, lengths, C_z, H_t, dtype, biases, in_place):
    z, w, out = _run(nt, lengths, C_z, H_t, dtype, biases, in_place=in_place)
    assert normwise_err(to_np(out), _ref(z, w), dtype=dtype) <= TOL[dtype]
    nt.nt_device_status()


def test_swiglu_full_size_sampled(nt):
    """The lognormal batch's 956,323 cells: sampled cells (first and last of
    every sample, and random ones) against the oracle."""
    cfg = wl.LOGNORMAL_BF16
    lengths = list(wl.draw_lengths(cfg, np.random.default_rng(0)))
    z, w, out = _run(nt, lengths, cfg.C_z, cfg.H_t, "bf16", biases=True)
    part = opart.partition(lengths)
    rng = np.random.default_rng(3)
    rows = np.concatenate([rng.integers(0, part.P, 3000), part.pair_off[:-1], part.pair_off[1:] - 1])
    got = to_np(out[torch.as_tensor(rows, device=DEV)])
    assert normwise_err(got, _ref(z, w, rows), dtype="bf16") <= TOL["bf16"]
    nt.nt_device_status()


def test_swiglu_zero_gate_is_residual_plus_bias(nt):
    """W1 = 0, b1 = 0 closes the gate: z~ = z + b2, rounded once to bf16."""
    lengths = [40, 7]
    part = nt.nt_partition_build(torch.as_tensor(np.asarray(lengths, dtype=np.int32)).to(DEV))
    P = opart.partition(lengths).P
    w = wl.make_swiglu_weights(128, 256, "bf16", biases=True, seed=4)
    z = wl.random_rows(P, 128, "bf16", seed=5).to(DEV)
    zero = torch.zeros_like(w.W1).to(DEV)
    out = nt.nt_pair_transition_swiglu(part, z, w.ln_gamma.to(DEV), w.ln_beta.to(DEV), zero, None, w.W3.to(DEV),
                                       w.b3.to(DEV), w.W2.to(DEV), w.b2.to(DEV))
    ref = (z.float() + w.b2.to(DEV)).to(torch.bfloat16)
    assert torch.equal(out, ref)
