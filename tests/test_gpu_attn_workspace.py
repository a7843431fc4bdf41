"""The attention calls keep their work counter in caller-owned workspace, so
launches that overlap on the GPU cannot take one another's work items.

Two packed streams with different inputs run at the same time on two CUDA
streams, eagerly and as two captured graphs replayed side by side.  Every
output must equal, bit for bit, what the same call gives when it runs alone
(each output row has exactly one owner, so the result does not depend on
which CTA takes which item), and must match the CPU oracle within the bf16
tolerance.  Without a workspace the call takes one CTA per item; its result
must be the same bits.
("Variable-length attention and data packing", "How to use it": one varlen
call per packed batch.)"""
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


def _problem(seed, total, lo, hi, H=4):
    rng = np.random.default_rng(seed)
    lens = wl.draw_segments(total, lo, hi, rng)
    a = wl.make_attn_inputs(wl.AttnConfig("ws", total, lo, hi, H, 64), seqlens=lens, seed=seed)
    cu = np.concatenate([[0], np.cumsum(lens.astype(np.int64))]).astype(np.int32)
    d = {"q": a.q.to(DEV), "k": a.k.to(DEV), "v": a.v.to(DEV), "cu": torch.as_tensor(cu).to(DEV),
         "max_len": int(lens.max()), "a": a, "cu_np": cu}
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty(H, d["q"].shape[0], dtype=torch.float32, device=DEV)
    d["ws"] = torch.empty(4096, dtype=torch.uint8, device=DEV)   # >= nt_varlen_attn_workspace_bytes()
    return d


def _call(nt, p, stream, workspace=None):
    nt.nt_varlen_attn(p["q"], p["k"], p["v"], p["cu"], p["max_len"], out=p["o"], lse=p["lse"], stream=stream,
                      workspace=p["ws"] if workspace is None else workspace)


def _oracle_check(p):
    a = p["a"]
    O_ref, lse_ref = oattn.varlen_attention(f64(a.q), f64(a.k), f64(a.v), p["cu_np"])
    assert normwise_err(to_np(p["o"]), O_ref, dtype="bf16") <= TOL["bf16"]
    assert np.abs(to_np(p["lse"]) - lse_ref).max() <= 2e-2


def test_workspace_size(nt):
    assert nt.nt_varlen_attn_workspace_bytes() >= 4
    assert nt.nt_varlen_attn_workspace_bytes() <= 4096


def test_concurrent_streams(nt):
    # short segments (mean <= 768 tokens): the persistent schedule with its counter
    pa = _problem(11, 6000, 16, 300)
    pb = _problem(12, 5000, 40, 500)
    s0 = torch.cuda.current_stream()
    _call(nt, pa, s0)
    _call(nt, pb, s0)
    torch.cuda.synchronize()
    ref_a = (pa["o"].clone(), pa["lse"].clone())
    ref_b = (pb["o"].clone(), pb["lse"].clone())
    _oracle_check(pa)
    _oracle_check(pb)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(8):
        pa["o"].zero_(); pb["o"].zero_()
        pa["lse"].zero_(); pb["lse"].zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(sa):
            _call(nt, pa, sa)
        with torch.cuda.stream(sb):
            _call(nt, pb, sb)
        torch.cuda.synchronize()
        assert torch.equal(pa["o"], ref_a[0]) and torch.equal(pa["lse"], ref_a[1]), f"stream A, repeat {rep}"
        assert torch.equal(pb["o"], ref_b[0]) and torch.equal(pb["lse"], ref_b[1]), f"stream B, repeat {rep}"
    nt.nt_device_status()


def test_graphs_replayed_side_by_side(nt):
    pa = _problem(21, 7000, 16, 512)
    pb = _problem(22, 4000, 16, 200)
    _call(nt, pa, torch.cuda.current_stream())
    _call(nt, pb, torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref_a, ref_b = pa["o"].clone(), pb["o"].clone()
    graphs = []
    for p in (pa, pb):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            _call(nt, p, s)                # warm-up on the capture stream
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                _call(nt, p, s)
        graphs.append(g)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(8):
        pa["o"].zero_(); pb["o"].zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(sa):
            graphs[0].replay()
        with torch.cuda.stream(sb):
            graphs[1].replay()
        torch.cuda.synchronize()
        assert torch.equal(pa["o"], ref_a), f"graph A, replay {rep}"
        assert torch.equal(pb["o"], ref_b), f"graph B, replay {rep}"
    _oracle_check(pa)
    _oracle_check(pb)
    nt.nt_device_status()


def test_no_workspace_same_bits(nt):
    p = _problem(31, 5000, 16, 512)
    _call(nt, p, torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref_o, ref_l = p["o"].clone(), p["lse"].clone()
    p["o"].zero_()
    p["lse"].zero_()
    _call(nt, p, torch.cuda.current_stream(), workspace=False)   # one CTA per item
    torch.cuda.synchronize()
    assert torch.equal(p["o"], ref_o) and torch.equal(p["lse"], ref_l)
    nt.nt_device_status()


def test_backward_concurrent_streams(nt):
    pa = _problem(41, 3000, 16, 300, H=2)
    pb = _problem(42, 2500, 16, 200, H=2)
    outs = []
    for p in (pa, pb):
        _call(nt, p, torch.cuda.current_stream())
        p["do"] = wl.random_rows(p["q"].shape[0] * 2, 64, wl.BF16, seed=5).reshape(p["q"].shape).to(DEV)
    torch.cuda.synchronize()
    for p in (pa, pb):
        outs.append(nt.nt_varlen_attn_bwd(p["q"], p["k"], p["v"], p["o"], p["do"], p["lse"], p["cu"], None,
                                          p["max_len"]))
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(4):
        res = []
        for p, s in ((pa, sa), (pb, sb)):
            with torch.cuda.stream(s):
                res.append(nt.nt_varlen_attn_bwd(p["q"], p["k"], p["v"], p["o"], p["do"], p["lse"], p["cu"], None,
                                                 p["max_len"], stream=s))
        torch.cuda.synchronize()
        for got, ref in zip(res, outs):
            for g_, r_ in zip(got, ref):
                assert torch.equal(g_, r_), f"backward, repeat {rep}"
    nt.nt_device_status()
