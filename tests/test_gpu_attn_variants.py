"""GPU parity of nt_varlen_attn_qk: causal self-attention and cross-attention
(separate query and key segments, "DanLing NestedTensor" section 3.3),
against the CPU oracle on the same seeded inputs.  Floats normwise,
max|gpu - oracle| / max|oracle| <= 2e-2 (bf16) or 1e-5 (fp32); queries that
see no key must come back as exact zeros with lse = -inf."""
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


def _run(nt, lq, lk, H, d, dtype, causal, seed=3):
    a = wl.make_cross_attn_inputs(lq, lk, H, d, dtype, seed=seed)
    cu_q, cu_k = _cu(lq), _cu(lk)
    o, l = nt.nt_varlen_attn_qk(a.q.to(DEV), a.k.to(DEV), a.v.to(DEV), torch.as_tensor(cu_q).to(DEV),
                                torch.as_tensor(cu_k).to(DEV), int(max(lq)), causal=causal, want_lse=True)
    O_ref, lse_ref = oattn.varlen_attention(f64(a.q), f64(a.k), f64(a.v), cu_q, causal=causal,
                                            cu_seqlens_k=cu_k)
    return a, o, l, O_ref, lse_ref


def _check(o, l, O_ref, lse_ref, dtype):
    o, l = to_np(o), to_np(l)
    dead = np.isneginf(lse_ref)                      # (H, T_q): queries that see no key
    assert np.array_equal(np.isneginf(l), dead)
    for h in range(dead.shape[0]):
        assert np.all(o[dead[h], h, :] == 0.0)
    assert normwise_err(o, O_ref, dtype=dtype) <= TOL[dtype]
    live = ~dead
    if live.any():
        assert np.abs(l[live] - lse_ref[live]).max() <= (1e-4 if dtype == "f32" else 2e-2)


@pytest.mark.parametrize("seqlens,H,d,dtype", [
    ([1, 63, 64, 65, 127, 128, 129, 300], 2, 64, "bf16"),   # tensor cores: every tile edge
    ([513, 2, 256], 3, 64, "bf16"),
    ([3, 1, 5, 0, 7, 64, 65, 130], 2, 64, "f32"),
    ([40, 9, 77], 2, 32, "f32"),
    ([40, 9, 77, 200], 2, 128, "bf16"),
    ([900, 1100], 2, 64, "bf16"),           # mean length > 768: one CTA per (segment, tile, head)
])
def test_causal_self_attention(nt, seqlens, H, d, dtype):
    a, o, l, O_ref, lse_ref = _run(nt, seqlens, seqlens, H, d, dtype, causal=True)
    _check(o, l, O_ref, lse_ref, dtype)
    # the first query of every segment sees only its own key: O = v exactly
    cu = _cu(seqlens)
    firsts = [int(cu[b]) for b in range(len(seqlens)) if seqlens[b] > 0]
    assert torch.equal(o[firsts].cpu(), a.v[firsts])
    nt.nt_device_status()


CROSS = [
    ([5, 0, 130, 64, 1, 200], [7, 3, 0, 64, 129, 150]),     # an empty key segment, an empty query segment
    ([256, 100], [40, 300]),
    ([130], [3]),                                           # causal: the first 127 queries see no key
    ([5, 70], [200, 64]),
    ([1000, 1200], [800, 1500]),                            # mean query length > 768: one CTA per item
]


@pytest.mark.parametrize("lq,lk", CROSS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cross_attention(nt, lq, lk, causal, dtype):
    _, o, l, O_ref, lse_ref = _run(nt, lq, lk, 2, 64, dtype, causal)
    _check(o, l, O_ref, lse_ref, dtype)
    nt.nt_device_status()


def test_no_keys_at_all(nt):
    """T_k = 0: every query sees nothing."""
    _, o, l, O_ref, lse_ref = _run(nt, [4, 9], [0, 0], 2, 64, "bf16", causal=False)
    assert torch.count_nonzero(o).item() == 0
    _check(o, l, O_ref, lse_ref, "bf16")
    nt.nt_device_status()


def test_self_through_qk_is_the_same_call(nt):
    """nt_varlen_attn and nt_varlen_attn_qk with cu_k = cu_q, causal = 0 give
    bit-identical results."""
    lens = [37, 128, 5, 200, 64]
    a = wl.make_cross_attn_inputs(lens, lens, 2, 64, "bf16", seed=5)
    cu = torch.as_tensor(_cu(lens)).to(DEV)
    q, k, v = a.q.to(DEV), a.k.to(DEV), a.v.to(DEV)
    o1, l1 = nt.nt_varlen_attn(q, k, v, cu, 200, want_lse=True)
    o2, l2 = nt.nt_varlen_attn_qk(q, k, v, cu, cu, 200, want_lse=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_cross_zero_leakage(nt):
    """Changing one segment's keys and values leaves every other segment's
    output bit-identical."""
    lq, lk = [37, 128, 5, 90], [60, 17, 200, 64]
    a = wl.make_cross_attn_inputs(lq, lk, 2, 64, "bf16", seed=6)
    cq, ck = torch.as_tensor(_cu(lq)).to(DEV), torch.as_tensor(_cu(lk)).to(DEV)
    q, k, v = a.q.to(DEV), a.k.to(DEV), a.v.to(DEV)
    o, _ = nt.nt_varlen_attn_qk(q, k, v, cq, ck, 128, causal=True)
    k2, v2 = k.clone(), v.clone()
    klo, khi = int(ck[2]), int(ck[3])
    k2[klo:khi] *= -3
    v2[klo:khi] = 7.0
    o2, _ = nt.nt_varlen_attn_qk(q, k2, v2, cq, ck, 128, causal=True)
    qlo, qhi = int(cq[2]), int(cq[3])
    assert torch.equal(o2[:qlo], o[:qlo]) and torch.equal(o2[qhi:], o[qhi:])
    assert not torch.equal(o2[qlo:qhi], o[qlo:qhi])


def test_causal_full_size_sampled(nt):
    """Causal self-attention over the packed stream of 65,536 tokens (237
    segments, 12 heads x 64): every output of a sample of segments against
    the oracle."""
    cfg = wl.VARLEN_ATTN_BF16
    a = wl.make_attn_inputs(cfg)
    cu = _cu(a.seqlens)
    cu_d = torch.as_tensor(cu).to(DEV)
    o, l = nt.nt_varlen_attn_qk(a.q.to(DEV), a.k.to(DEV), a.v.to(DEV), cu_d, cu_d, int(a.seqlens.max()),
                                causal=True, want_lse=True)
    B = len(a.seqlens)
    segs = sorted(set([0, B - 1, int(np.argmax(a.seqlens)), int(np.argmin(a.seqlens))] +
                      list(np.random.default_rng(4).integers(0, B, size=6))))
    O_ref, lse_ref = oattn.varlen_attention(f64(a.q), f64(a.k), f64(a.v), cu, segments=segs, causal=True)
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in segs])
    idx = torch.as_tensor(rows, device=DEV)
    assert normwise_err(to_np(o[idx]), O_ref[rows], dtype="bf16") <= TOL["bf16"]
    assert np.abs(to_np(l[:, idx]) - lse_ref[:, rows]).max() <= 2e-2
    nt.nt_device_status()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bad_key_offsets_flagged(nt, dtype):
    """Key offsets whose last entry exceeds T_k are caught by the kernels'
    own bounds checks (status word), with no access beyond the buffers."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.zeros(64, 1, 64, dtype=tdt, device=DEV)
    k = torch.zeros(32, 1, 64, dtype=tdt, device=DEV)
    cu_q = torch.tensor([0, 32, 64], dtype=torch.int32, device=DEV)
    cu_k = torch.tensor([0, 16, 48], dtype=torch.int32, device=DEV)
    nt.nt_varlen_attn_qk(q, k, k, cu_q, cu_k, 32)
    with pytest.raises(nt.NTError) as ei:
        nt.nt_device_status()
    assert ei.value.status == 6
