"""nt_pair_broadcast_noalloc, the pair broadcast for callers that cannot
allocate device memory (a plug-in whose host framework owns every device
allocation, or a real-time loop that must not allocate on its hot path).

It must give the same pair cells as nt_pair_broadcast with a caller
workspace, call after call, even though every call reuses the library's one
built-in scratch array.  The test drives the C ABI directly (ctypes) and
allocates every input and output itself before the calls.
"""
import ctypes

import numpy as np
import pytest
import torch

from _helpers import TOL, f64, normwise_err, to_np
from oracle import block as oblock
from variable_length_batching_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"
LIMIT = 2 * 1024 * 1024      # fp32 elements of the built-in scratch: (T + T_cols) * C_z


@pytest.fixture(scope="module")
def nt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_batching_gb300 import build, nt as ntmod
    build.build()
    return ntmod


def _noalloc(nt, part, s_left, s_right, W_a, W_b, z):
    L = nt.lib()
    return L.nt_pair_broadcast_noalloc(ctypes.byref(part.c), nt.NT_BF16, ctypes.c_void_p(s_left.data_ptr()),
                                       ctypes.c_void_p(s_right.data_ptr()), s_left.shape[1],
                                       ctypes.c_void_p(W_a.data_ptr()), ctypes.c_void_p(W_b.data_ptr()),
                                       W_a.shape[0], ctypes.c_void_p(z.data_ptr()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_call_twice(nt):
    """Two different batches in a row: the second call must not see the
    first's scratch.  Both calls run the same kernels with the same roundings
    as the workspace call, so the cells must be bit-identical; they must
    also match the CPU oracle."""
    cfg = wl.PAIRFORMER_BF16
    for seed, lengths in ((0, None), (1, [3, 250, 1, 0, 77])):
        inp = wl.make_block_inputs(cfg, lengths=lengths, seed=seed)
        w = inp.blocks[0]
        part = nt.nt_partition_build(torch.as_tensor(inp.lengths).to(DEV))
        assert 2 * part.T * cfg.C_z <= LIMIT
        s, W_a, W_b = inp.s.to(DEV), w.W_a.to(DEV), w.W_b.to(DEV)
        z_ref = nt.nt_pair_broadcast(part, s, s, W_a, W_b)
        z = torch.full_like(z_ref, float("nan"))
        assert _noalloc(nt, part, s, s, W_a, W_b, z) == 0, nt.lib().nt_last_error()
        torch.cuda.synchronize()
        assert torch.equal(z, z_ref)
        ref = oblock.pair_broadcast(inp.lengths, f64(inp.s), f64(inp.s), f64(w.W_a), f64(w.W_b))
        assert normwise_err(to_np(z), ref, dtype="bf16") <= TOL["bf16"]
        nt.nt_device_status()


def test_noalloc_rectangular_at_the_limit(nt):
    """A rectangular batch (T_cols != T) whose u and v fill the scratch to
    within a few rows of its size, so v's place in it is exercised at the
    limit; called twice in a row with different singles."""
    cfg = wl.RECT_BF16
    C_z = cfg.C_z
    rows = [40, 1, 0, 97, 63, 200, 33, 18] * 8            # T = 3,616
    cols = [300, 1, 380, 0, 200, 360, 171, 180] * 8      # T_cols = 12,736
    T, T_cols = sum(rows), sum(cols)
    assert (T + T_cols) * C_z <= LIMIT and (T + T_cols + 64) * C_z > LIMIT
    for seed in (3, 4):
        inp = wl.make_rect_inputs(cfg, rows=rows, cols=cols, seed=seed)
        w = inp.blocks[0]
        part = nt.nt_partition_build_rect(torch.as_tensor(inp.rows).to(DEV), torch.as_tensor(inp.cols).to(DEV))
        sr, sc, W_a, W_b = inp.s_row.to(DEV), inp.s_col.to(DEV), w.W_a.to(DEV), w.W_b.to(DEV)
        ws = torch.empty(nt.nt_pair_broadcast_workspace_bytes_rect(part.T, part.T_cols, C_z), dtype=torch.uint8,
                         device=DEV)
        z_ref = torch.empty(part.P, C_z, dtype=torch.bfloat16, device=DEV)
        nt.nt_pair_broadcast(part, sr, sc, W_a, W_b, z=z_ref, workspace=ws)
        z = torch.full_like(z_ref, float("nan"))
        assert _noalloc(nt, part, sr, sc, W_a, W_b, z) == 0, nt.lib().nt_last_error()
        torch.cuda.synchronize()
        assert torch.equal(z, z_ref)
        ref = oblock.pair_broadcast_rect(inp.rows, inp.cols, f64(inp.s_row), f64(inp.s_col), f64(w.W_a),
                                         f64(w.W_b))
        assert normwise_err(to_np(z), ref, dtype="bf16") <= TOL["bf16"]
        nt.nt_device_status()


def test_noalloc_rejects_beyond_limit(nt):
    """A batch whose u and v would not fit the built-in scratch is refused
    with NT_ERR_UNSUPPORTED before anything is enqueued."""
    cfg = wl.PAIRFORMER_BF16
    lengths = [1] * (LIMIT // (2 * cfg.C_z) + 1)
    part = nt.nt_partition_build(torch.as_tensor(np.asarray(lengths, dtype=np.int32)).to(DEV))
    s = torch.zeros(part.T, cfg.C_s, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(cfg.C_z, cfg.C_s, dtype=torch.bfloat16, device=DEV)
    z = torch.zeros(part.P, cfg.C_z, dtype=torch.bfloat16, device=DEV)
    assert _noalloc(nt, part, s, s, W, W, z) == 2
    assert b"scratch" in nt.lib().nt_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(z) == 0
