"""Device-side failure reporting on the GPU, without a fault: the bounded
mbarrier wait that every tensor-core kernel uses, driven through its three
outcomes by nt_selftest_bounded_wait.  A wait that runs out is reported once
by nt_device_status as NT_ERR_TIMEOUT, and the context still computes a
block that matches the oracle afterwards."""
import numpy as np
import pytest
import torch

from _helpers import TOL, f64, normwise_err, oracle_weights, to_np
from oracle import block as oblock
from variable_length_batching_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
MS = 10 ** 6


@pytest.fixture(scope="module")
def nt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_batching_gb300 import build, nt as ntmod
    build.build()
    return ntmod


def _block_matches_oracle(nt):
    inp = wl.make_block_inputs(wl.PAIRFORMER_BF16, lengths=[37, 1, 0, 70], biases=True)
    w = inp.blocks[0]
    dw = lambda t: None if t is None else t.to(DEV).contiguous()
    from types import SimpleNamespace
    ws = SimpleNamespace(**{k: dw(getattr(w, k)) for k in ("W_a", "W_b", "ln_gamma", "ln_beta", "W1", "b1", "W2",
                                                         "b2", "W_g", "b_g")})
    part = nt.nt_partition_build(torch.as_tensor(np.asarray(inp.lengths, dtype=np.int32)).to(DEV))
    z, m, s_out = nt.block_forward(part, inp.s.to(DEV), ws)
    assert nt.nt_device_status() == 0
    ref = oblock.block_packed(inp.lengths, f64(inp.s), oracle_weights(w))
    assert normwise_err(to_np(z), ref.z_tilde, dtype="bf16") <= TOL["bf16"]
    assert normwise_err(to_np(s_out), ref.s_out, dtype="bf16") <= TOL["bf16"]


def test_wait_completes(nt):
    r = nt.nt_selftest_bounded_wait(0, 2 * MS, 1000 * MS)
    assert nt.nt_device_status() == 0
    ok, dur = r.tolist()
    assert ok == 1
    assert 1 * MS <= dur < 500 * MS, dur


def test_wait_runs_out_and_is_reported_once(nt):
    r = nt.nt_selftest_bounded_wait(1, 0, 20 * MS)
    with pytest.raises(nt.NTError) as err:
        nt.nt_device_status()
    assert err.value.status == 5                 # NT_ERR_TIMEOUT
    ok, dur = r.tolist()
    assert ok == 0
    assert 20 * MS <= dur < 1000 * MS, dur
    assert nt.nt_device_status() == 0            # read once, then cleared
    _block_matches_oracle(nt)                    # the context is still usable


def test_abort_flag_ends_the_wait_without_flagging(nt):
    r = nt.nt_selftest_bounded_wait(2, 2 * MS, 1000 * MS)
    assert nt.nt_device_status() == 0
    ok, dur = r.tolist()
    assert ok == 0
    assert 1 * MS <= dur < 500 * MS, dur
