"""One single -> pair -> single block step ("DanLing NestedTensor" Eq. 1) with
host inputs and outputs, replayed from a CUDA graph.

Each step copies the sample lengths and the singles in from pinned host
memory and rebuilds the partition in one call (its totals come back to the
host: they decide the pair state's size).  Everything after that has fixed sizes for a
given (B, T, P) and runs as one captured graph: the broadcast, the
transition in slices of cells of growing length (each slice's z~ copied
back to the host on a second stream as soon as it is done, so the read-back
overlaps the next slice), the reduce, and the copy-back of s_out.  A new (B, T, P) captures a
new graph.  Every device step runs in the library's kernels; this module
only owns the buffers, the streams and the graph.
"""
import ctypes
from typing import List, Optional

import torch

from . import nt as _nt


def slice_cuts(P: int, slices: int, growth: float = 1.0) -> List[int]:
    """Cell boundaries of ``slices`` consecutive ranges covering [0, P), each
    ``growth`` times as long as the one before (up to rounding).  A small
    first range lets the first read-back start early; the later, longer
    ones are transformed while the host link drains the earlier ones."""
    if slices < 1 or growth <= 0:
        raise ValueError("slices must be >= 1 and growth > 0")
    w = [growth ** i for i in range(slices)]
    tot = sum(w)
    cuts, acc = [0], 0.0
    for x in w[:-1]:
        acc += x
        cuts.append(min(P, max(cuts[-1], int(round(P * acc / tot)))))
    cuts.append(P)
    return cuts


class BlockGraph:
    """Host-to-host block steps for fixed weights ``w`` (a namespace of device
    tensors W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, b2, W_g, b_g; bf16 or
    fp32 like the singles).  The transition runs in ``slices`` cell ranges,
    each ``growth`` times as long as the one before."""

    def __init__(self, w, slices: int = 3, growth: float = 2.0, ln_eps: float = 1e-5,
                 device: Optional[torch.device] = None):
        if slices < 1 or growth <= 0:
            raise ValueError("slices must be >= 1 and growth > 0")
        self.w = w
        self.slices = slices
        self.growth = growth
        self.ln_eps = ln_eps
        self.dev = device if device is not None else w.W_a.device
        self.C_z, self.C_s = w.W_a.shape
        self.copy_stream = torch.cuda.Stream(device=self.dev)
        self.graph = None
        self.key = None
        self.B = -1
        self.T = -1

    # -- static buffers --------------------------------------------------------------
    def _ensure_b(self, B: int):
        if B == self.B:
            return
        self.B = B
        self.lengths = torch.empty(B, dtype=torch.int32, device=self.dev)
        self.cu = torch.empty(B + 1, dtype=torch.int32, device=self.dev)
        self.pair_off = torch.empty(B + 1, dtype=torch.int64, device=self.dev)
        self.totals = torch.empty(4, dtype=torch.int64, device=self.dev)
        self.key = None

    def _ensure_t(self, T: int, dtype: torch.dtype):
        if T == self.T and getattr(self, "s", None) is not None and self.s.dtype == dtype:
            return
        self.T = T
        self.s = torch.empty(T, self.C_s, dtype=dtype, device=self.dev)
        self.row_start = torch.empty(T + 1, dtype=torch.int64, device=self.dev)
        self.row_sample = torch.empty(max(T, 1), dtype=torch.int32, device=self.dev)
        self.key = None

    def _partition(self, stream) -> "_nt.Partition":
        # scan and row splits in one call (the singles' row count bounds T)
        c = _nt.nt_partition()
        st = _nt.lib().nt_partition_build_with_rows(
            _nt._ptr(self.lengths) if self.B else None, self.B, self.T, _nt._ptr(self.cu), _nt._ptr(self.pair_off),
            _nt._ptr(self.totals), _nt._ptr(self.row_start), _nt._ptr(self.row_sample), ctypes.byref(c),
            _nt._stream(stream))
        _nt._check(st, "nt_partition_build_with_rows")
        if c.T != self.T:
            raise ValueError(f"the lengths sum to {c.T}, the singles have {self.T} rows")
        return _nt.Partition(self.lengths, self.cu, self.pair_off, self.totals, self.row_start, self.row_sample, c)

    # -- the captured part ---------------------------------------------------------
    def _body(self, part):
        w = self.w
        main = torch.cuda.current_stream(self.dev)
        _nt.nt_pair_broadcast(part, self.s, self.s, w.W_a, w.W_b, z=self.z, workspace=self.ws)
        P = part.P
        cuts = slice_cuts(P, self.slices, self.growth)
        for c0, c1 in zip(cuts[:-1], cuts[1:]):
            if c1 == c0:
                continue
            _nt.nt_pair_transition_cells(self.z[c0:c1], w.ln_gamma, w.ln_beta, w.W1, w.b1, w.W2, w.b2,
                                         ln_eps=self.ln_eps, out=self.z[c0:c1])
            self.copy_stream.wait_stream(main)
            with torch.cuda.stream(self.copy_stream):
                self.z_host[c0:c1].copy_(self.z[c0:c1], non_blocking=True)
        _nt.nt_pair_reduce(part, self.z, w.W_g, w.b_g, s_in=self.s, m=self.m, s_out=self.s_out)
        self.s_out_host.copy_(self.s_out, non_blocking=True)
        main.wait_stream(self.copy_stream)

    def _capture(self, part, dtype):
        P, T = part.P, part.T
        self.z = torch.empty(P, self.C_z, dtype=dtype, device=self.dev)
        self.m = torch.empty(T, self.C_z, dtype=dtype, device=self.dev)
        self.s_out = torch.empty(T, self.C_s, dtype=dtype, device=self.dev)
        need = _nt.nt_pair_broadcast_workspace_bytes_rect(T, T, self.C_z)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=self.dev)
        self.z_host = torch.empty(P, self.C_z, dtype=dtype).pin_memory()
        self.s_out_host = torch.empty(T, self.C_s, dtype=dtype).pin_memory()
        # one eager pass first (launch attributes, tensor maps, the library's
        # own lazy set-up happen outside the capture)
        self._body(part)
        torch.cuda.synchronize(self.dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._body(part)
        self.key = (self.B, T, P)

    def run(self, lengths_host: torch.Tensor, s_host: torch.Tensor):
        """One step: ``lengths_host`` (int32, B) and ``s_host`` (T x C_s), both
        in pinned host memory.  Returns pinned host tensors (z~ of P x C_z,
        s_out of T x C_s), overwritten by the next call."""
        if lengths_host.dtype != torch.int32 or s_host.dim() != 2 or s_host.shape[1] != self.C_s:
            raise ValueError("lengths must be int32 (B,) and s (T, C_s)")
        main = torch.cuda.current_stream(self.dev)
        self._ensure_b(lengths_host.numel())
        self._ensure_t(s_host.shape[0], s_host.dtype)
        self.lengths.copy_(lengths_host, non_blocking=True)
        self.s.copy_(s_host, non_blocking=True)
        part = self._partition(main)
        if self.key != (self.B, part.T, part.P):
            self._capture(part, s_host.dtype)
        else:
            self.graph.replay()
        main.synchronize()
        return self.z_host, self.s_out_host
