"""GPU parity of the varlen attention backward (nt_varlen_attn_bwd): dq, dk,
dv for an upstream gradient, against the CPU oracle's gradients on the same
seeded inputs.  The forward outputs the backward consumes (o and the
natural-log lse) come from the oracle too, so no expected value or input
passes through the CUDA path.  Normwise tolerance: 2e-2 bf16, 1e-5 fp32."""
import numpy as np
import pytest
import torch

from _helpers import TOL, f64, normwise_err, to_np
from oracle import attention as oattn
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


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def _case(nt, lq, lk, H, d, dtype, causal, segments=None, seed=7):
    a = wl.make_cross_attn_inputs(lq, lk, H, d, dtype, seed=seed)
    do = wl.random_rows(int(sum(lq)) * H, d, dtype, seed=seed + 1).reshape(int(sum(lq)), H, d)
    cu_q, cu_k = _cu(lq), _cu(lk)
    cross = None if list(lq) == list(lk) else cu_k
    q, k, v, g = f64(a.q), f64(a.k), f64(a.v), f64(do)
    O, L = oattn.varlen_attention(q, k, v, cu_q, causal=causal, cu_seqlens_k=cross, segments=segments)
    dq_r, dk_r, dv_r = oattn.varlen_attention_backward(q, k, v, g, cu_q, causal=causal, cu_seqlens_k=cross,
                                                       segments=segments)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    o_in = torch.from_numpy(O).to(tdt).to(DEV)
    lse_in = torch.from_numpy(L.astype(np.float32)).to(DEV)
    dq, dk, dv = nt.nt_varlen_attn_bwd(a.q.to(DEV), a.k.to(DEV), a.v.to(DEV), o_in, do.to(DEV), lse_in,
                                       torch.as_tensor(cu_q).to(DEV), torch.as_tensor(cu_k).to(DEV),
                                       max(list(lq) + [0]), max(list(lk) + [0]), causal=causal)
    return (dq, dk, dv), (dq_r, dk_r, dv_r), cu_q, cu_k


@pytest.mark.parametrize("lq,lk,H,d,dtype,causal", [
    ([3, 1, 5, 0, 7, 64, 65, 130], None, 2, 64, "bf16", False),
    ([3, 1, 5, 0, 7, 64, 65, 130], None, 2, 64, "bf16", True),
    ([40, 9, 77], None, 2, 32, "f32", False),
    ([40, 9, 77], None, 2, 64, "f32", True),
    ([20, 33], None, 2, 128, "f32", False),
    ([5, 0, 130, 64, 1, 200], [7, 3, 0, 64, 129, 150], 2, 64, "bf16", True),   # cross, empty and all-masked rows
    ([130], [3], 2, 64, "f32", True),                                          # 127 queries see no key
    ([130], [3], 2, 64, "bf16", True),
    ([3, 300], [200, 17], 3, 64, "bf16", False),                              # cross: 5 key tiles / 1 query tile
    ([511, 1, 256, 129], None, 2, 64, "bf16", True),                           # several 128-key and 64-query tiles
    ([511, 1, 256, 129], None, 2, 64, "bf16", False),
    ([1000, 1300], None, 2, 64, "bf16", False),                               # mean > 768: one CTA per item
    ([1000, 1300], None, 2, 64, "bf16", True),
    ([900, 1000], [1200, 700], 2, 64, "bf16", True),
    ([1, 2000, 3, 0, 5, 2, 1, 7, 9, 400], None, 1, 64, "bf16", True),          # persistent, mostly empty tiles
])
def test_attention_backward(nt, lq, lk, H, d, dtype, causal):
    lk = lq if lk is None else lk
    got, ref, _, _ = _case(nt, lq, lk, H, d, dtype, causal)
    for g, r in zip(got, ref):
        assert normwise_err(to_np(g), r, dtype=dtype) <= TOL[dtype]
    nt.nt_device_status()


@pytest.mark.parametrize("causal", [True, False])
def test_attention_backward_full_size_sampled(nt, causal):
    """The 65,536-token stream (237 segments, 12 heads x 64): every gradient
    row of a sample of segments against the oracle."""
    a = wl.make_attn_inputs(wl.VARLEN_ATTN_BF16)
    lens = list(a.seqlens)
    B = len(lens)
    segs = sorted(set([0, B - 1, int(np.argmax(a.seqlens)), int(np.argmin(a.seqlens)), 17, 101]))
    got, ref, cu, _ = _case(nt, lens, lens, 12, 64, "bf16", causal, segments=segs, seed=0)
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in segs])
    idx = torch.as_tensor(rows, device=DEV)
    for g, r in zip(got, ref):
        assert normwise_err(to_np(g[idx]), r[rows], dtype="bf16") <= TOL["bf16"]
    nt.nt_device_status()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_attention_backward_bad_cu_flagged(nt, dtype):
    """Offsets whose last entry exceeds T are caught by the kernels' own
    bounds checks (status word, NT_ERR_DEVICE_CHECK), with no access beyond
    the buffers, on the tensor-core (bf16) and CUDA-core (fp32) paths."""
    T, H, d = 64, 1, 64
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = torch.zeros(T, H, d, dtype=tdt, device=DEV)
    lse = torch.zeros(H, T, dtype=torch.float32, device=DEV)
    cu_bad = torch.tensor([0, 32, 96], dtype=torch.int32, device=DEV)
    nt.nt_varlen_attn_bwd(x, x, x, x, x, lse, cu_bad, None, 64)
    with pytest.raises(nt.NTError) as ei:
        nt.nt_device_status()
    assert ei.value.status == 6


def test_attention_backward_understated_max_len_flagged(nt):
    """A longest segment longer than the stated max_len is reported
    (NT_ERR_DEVICE_CHECK) instead of leaving gradient rows silently unwritten."""
    lens = [200, 10]
    a = wl.make_cross_attn_inputs(lens, lens, 2, 64, "bf16", seed=3)
    q, k, v = a.q.to(DEV), a.k.to(DEV), a.v.to(DEV)
    cu = torch.as_tensor(_cu(lens)).to(DEV)
    o, lse = nt.nt_varlen_attn_qk(q, k, v, cu, cu, max(lens), want_lse=True)
    nt.nt_device_status()
    nt.nt_varlen_attn_bwd(q, k, v, o, torch.ones_like(o), lse, cu, None, 64)
    with pytest.raises(nt.NTError) as ei:
        nt.nt_device_status()
    assert ei.value.status == 6
