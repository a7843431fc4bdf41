"""GPU parity of nt_pair_transition_cells: the transition run slice by
slice over a pair state (the form that lets finished slices be read back
while the next one computes) equals the whole-state call cell for cell, bit
for bit ("DanLing NestedTensor" section 3.3: the transition maps each valid
cell on its own), for the tensor-core ReLU and SwiGLU kernels and the fp32
CUDA-core kernel."""
import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("cfg,glu", [(wl.PAIRFORMER_BF16, False), (wl.PAIRFORMER_BF16, True),
                                     (wl.TINY_FP32, False)])
def test_transition_by_slices_equals_whole(nt, cfg, glu):
    inp = wl.make_block_inputs(cfg, biases=True)
    w = inp.blocks[0]
    g = lambda t: None if t is None else t.to(DEV).contiguous()
    part = nt.nt_partition_build(_dev(inp.lengths))
    s = inp.s.to(DEV)
    z = nt.nt_pair_broadcast(part, s, s, g(w.W_a), g(w.W_b))
    W1, b1, W2, b2, W3, b3 = g(w.W1), g(w.b1), g(w.W2), g(w.b2), None, None
    if glu:
        sw = wl.make_swiglu_weights(cfg.C_z, cfg.H_t, cfg.dtype, biases=True, seed=4)
        W1, b1, W2, b2, W3, b3 = g(sw.W1), g(sw.b1), g(sw.W2), g(sw.b2), g(sw.W3), g(sw.b3)
    gamma, beta = g(w.ln_gamma), g(w.ln_beta)
    if glu:
        whole = nt.nt_pair_transition_swiglu(part, z, gamma, beta, W1, b1, W3, b3, W2, b2)
    else:
        whole = nt.nt_pair_transition(part, z, gamma, beta, W1, b1, W2, b2)
    P = part.P
    cuts = sorted(set([0, 1, 300, min(4097, P), P // 2, P]))
    out = torch.empty_like(z)
    for c0, c1 in zip(cuts[:-1], cuts[1:]):
        nt.nt_pair_transition_cells(z[c0:c1], gamma, beta, W1, b1, W2, b2, W3=W3, b3=b3, out=out[c0:c1])
    assert torch.equal(out, whole)
    # zero cells: a no-op
    nt.nt_pair_transition_cells(z[:0], gamma, beta, W1, b1, W2, b2, W3=W3, b3=b3, out=out[:0])
    nt.nt_device_status()


# Cell counts around the tensor-core transition's work units (128-row
# sub-tiles; full 256-row tiles in whole waves of the grid, then half tiles
# when the rest fits in one more wave, else full tiles only; at most one
# sub-tile per SM: one half tile per CTA), for a 152-SM grid.
UNIT_CASES = [
    152 * 256,                    # whole waves of full tiles, no half tile
    152 * 256 + 11 * 128,         # one wave and 11 half tiles
    152 * 256 + 11 * 128 - 5,     # the same, the last half tile ragged
    2 * 152 * 256 + 153 * 128 + 1,  # the rest exceeds one wave: full tiles only
    152 * 128 + 1,                # one sub-tile past "one per SM"
]


@pytest.mark.parametrize("P", UNIT_CASES)
def test_transition_work_units(nt, P):
    """The tensor-core transition at cell counts that cut its work units in
    each way: sampled cells against the oracle, and in place equal to out
    of place bit for bit."""
    from _helpers import TOL, f64, normwise_err, to_np
    from oracle import block as oblock
    cfg = wl.PAIRFORMER_BF16
    w = wl.make_block_inputs(cfg, lengths=[1], biases=True).blocks[0]
    g = lambda t: None if t is None else t.to(DEV).contiguous()
    z = wl.random_rows(P, cfg.C_z, cfg.dtype, seed=P % 1000, scale=1.5).to(DEV)
    out = nt.nt_pair_transition_cells(z, g(w.ln_gamma), g(w.ln_beta), g(w.W1), g(w.b1), g(w.W2), g(w.b2))
    zi = z.clone()
    nt.nt_pair_transition_cells(zi, g(w.ln_gamma), g(w.ln_beta), g(w.W1), g(w.b1), g(w.W2), g(w.b2), out=zi)
    torch.cuda.synchronize()
    nt.nt_device_status()
    assert torch.equal(zi, out)
    rng = np.random.default_rng(P)
    idx = np.unique(np.concatenate([rng.integers(0, P, 500), np.arange(max(0, P - 12), P)]))
    zs = f64(z[torch.as_tensor(idx, device=DEV)].cpu())
    ref = oblock.pair_transition(zs, f64(w.ln_gamma), f64(w.ln_beta), 1e-5, f64(w.W1), f64(w.b1), f64(w.W2),
                                 f64(w.b2))
    got = to_np(out[torch.as_tensor(idx, device=DEV)])
    assert normwise_err(got, ref, dtype="bf16") <= TOL["bf16"]
