"""One single -> pair -> single block step ("DanLing NestedTensor" Eq. 1) with
host inputs and outputs, replayed from CUDA graphs, and consecutive steps
pipelined.

Each step copies the sample lengths and the singles in from pinned host
memory and rebuilds the partition in one call (its totals come back to the
host: they decide the pair state's size).  Everything after that has fixed
sizes for a given (B, T, P) and runs as captured graphs, one per slice of
cells: the first holds the broadcast and the first transition slice, the
last the last slice and the reduce.  Slices grow in length; each slice's z~
is copied back to the host on a second stream as soon as its graph is done,
then s_out.

Steps are pipelined over ``depth`` slots used in turn.  A slot holds the
step's device inputs (lengths, singles, the partition built from them), the
device buffers it writes (z~, m, s_out), the host buffers it fills and its
graphs.  The next step's copies in and partition run on an input stream of
their own while the current step's graphs run, and its graphs run while the
host link still drains the previous step's read-backs.  A slot's inputs are
overwritten only after its previous graphs have read them, and its outputs
only after their last read-back has completed.  A new (B, T, P) drains the
pipeline and captures new graphs.  Every device step runs in the library's
kernels; this module owns the buffers, the streams, the events and the
graphs.
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


class _Inputs:
    """Device inputs of one pipeline slot: the lengths, the singles and the
    partition built from them."""

    def __init__(self, B: int, T: int, C_s: int, dtype: torch.dtype, dev):
        self.lengths = torch.empty(B, dtype=torch.int32, device=dev)
        self.cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
        self.pair_off = torch.empty(B + 1, dtype=torch.int64, device=dev)
        self.totals = torch.empty(4, dtype=torch.int64, device=dev)
        self.s = torch.empty(T, C_s, dtype=dtype, device=dev)
        self.row_start = torch.empty(T + 1, dtype=torch.int64, device=dev)
        self.row_sample = torch.empty(max(T, 1), dtype=torch.int32, device=dev)
        self.part = None
        self.ready = torch.cuda.Event()    # input stream: copies and partition done
        self.free = torch.cuda.Event()     # main stream: the slot's last graph has read them
        self.used = False


class _Set:
    """Output buffers, graphs and events of one pipeline slot."""

    def __init__(self):
        self.graphs = []
        self.sliced = []        # event per slice, recorded on the main stream after its graph
        self.done = None        # recorded on the copy stream after the step's last read-back
        self.busy = False
        self.ticket = -1


class BlockGraph:
    """Host-to-host block steps for fixed weights ``w`` (a namespace of device
    tensors W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, b2, W_g, b_g; bf16 or
    fp32 like the singles).  ``readback`` chooses what a step returns to the
    host: "pair", the pair output z~ and s_out (the transition then runs in
    ``slices`` cell ranges, each ``growth`` times as long as the one before,
    so that each range's z~ is read back while the next one computes), or
    "loss", the Eq. 5 loss of the step's two outputs, computed on the device
    ("DanLing NestedTensor" Appendix A.1), and s_out (z~ stays on the
    device; one range).  ``depth`` steps may be in flight at once
    (``submit`` / ``wait``)."""

    def __init__(self, w, slices: int = 3, growth: float = 2.0, depth: int = 2, ln_eps: float = 1e-5,
                 device: Optional[torch.device] = None, readback: str = "pair"):
        if slices < 1 or growth <= 0 or depth < 1:
            raise ValueError("slices and depth must be >= 1, growth > 0")
        if readback not in ("pair", "loss"):
            raise ValueError("readback must be 'pair' or 'loss'")
        self.readback = readback
        if readback == "loss":
            slices = 1
        self.w = w
        self.slices = slices
        self.growth = growth
        self.depth = depth
        self.ln_eps = ln_eps
        self.dev = device if device is not None else w.W_a.device
        self.C_z, self.C_s = w.W_a.shape
        self.copy_stream = torch.cuda.Stream(device=self.dev)
        self.in_stream = torch.cuda.Stream(device=self.dev)
        self.key = None
        self.sets: List[_Set] = []
        self.retired = {}        # ticket -> slot of a step submitted before a shape change, until waited
        self.inputs: List[_Inputs] = []
        self.in_key = None
        self.submitted = 0

    # -- input slots --------------------------------------------------------------
    def _ensure_inputs(self, B: int, T: int, dtype: torch.dtype):
        if self.in_key == (B, T, dtype):
            return
        self._drain()            # in-flight steps still read the old input buffers
        self.inputs = [_Inputs(B, T, self.C_s, dtype, self.dev) for _ in range(self.depth)]
        self.in_key = (B, T, dtype)
        self.key = None          # the graphs capture the input buffers' addresses

    def _partition(self, inp: _Inputs, B: int, T: int, stream) -> "_nt.Partition":
        # scan and row splits in one call (the singles' row count bounds T);
        # the totals' read-back synchronises `stream` only
        c = _nt.nt_partition()
        st = _nt.lib().nt_partition_build_with_rows(
            _nt._ptr(inp.lengths) if B else None, B, T, _nt._ptr(inp.cu), _nt._ptr(inp.pair_off),
            _nt._ptr(inp.totals), _nt._ptr(inp.row_start), _nt._ptr(inp.row_sample), ctypes.byref(c),
            _nt._stream(stream))
        _nt._check(st, "nt_partition_build_with_rows")
        if c.T != T:
            raise ValueError(f"the lengths sum to {c.T}, the singles have {T} rows")
        return _nt.Partition(inp.lengths, inp.cu, inp.pair_off, inp.totals, inp.row_start, inp.row_sample, c)

    # -- the captured parts ------------------------------------------------------------
    def _piece(self, k: int, idx: int):
        """Slice ``idx`` of slot ``k``'s step: the broadcast before the first
        slice, the reduce after the last."""
        w = self.w
        st = self.sets[k]
        inp = self.inputs[k]
        part = inp.part
        c0, c1 = self.cuts[idx], self.cuts[idx + 1]
        if idx == 0:
            _nt.nt_pair_broadcast(part, inp.s, inp.s, w.W_a, w.W_b, z=st.z, workspace=self.ws)
        if c1 > c0:
            _nt.nt_pair_transition_cells(st.z[c0:c1], w.ln_gamma, w.ln_beta, w.W1, w.b1, w.W2, w.b2,
                                         ln_eps=self.ln_eps, out=st.z[c0:c1])
        if idx == self.slices - 1:
            if self.readback == "loss":      # the reduce reads z~ once for the mean and the loss
                _nt.nt_pair_reduce_loss(part, st.z, w.W_g, w.b_g, s_in=inp.s, m=st.m, s_out=st.s_out, loss=st.loss,
                                        workspace=self.loss_ws)
            else:
                _nt.nt_pair_reduce(part, st.z, w.W_g, w.b_g, s_in=inp.s, m=st.m, s_out=st.s_out)

    def _drain(self):
        for st in self.sets:
            if st.busy:
                st.done.synchronize()
                st.busy = False
        torch.cuda.synchronize(self.dev)
        for inp in self.inputs:
            inp.used = False

    def _setup(self, part, dtype):
        """Output buffers for a new (B, T, P); graphs are captured on each slot's first use.
        The old slots of steps not yet waited on keep their host results
        (their device work has drained) until ``wait`` collects them."""
        self._drain()
        for st in self.sets:
            if st.ticket >= 0 and st.ticket >= self.submitted - self.depth:
                self.retired[st.ticket] = st
        for t in [t for t in self.retired if t < self.submitted - self.depth]:
            del self.retired[t]
        P, T = part.P, part.T
        self.cuts = slice_cuts(P, self.slices, self.growth)
        need = _nt.nt_pair_broadcast_workspace_bytes_rect(T, T, self.C_z)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device=self.dev)
        self.loss_ws = torch.empty(max(int(_nt.lib().nt_pair_reduce_loss_workspace_bytes()), 16),
                                   dtype=torch.uint8, device=self.dev)
        self.sets = []
        for _ in range(self.depth):
            st = _Set()
            st.z = torch.empty(P, self.C_z, dtype=dtype, device=self.dev)
            st.m = torch.empty(T, self.C_z, dtype=dtype, device=self.dev)
            st.s_out = torch.empty(T, self.C_s, dtype=dtype, device=self.dev)
            if self.readback == "pair":
                st.z_host = torch.empty(P, self.C_z, dtype=dtype).pin_memory()
            else:
                st.loss = torch.empty(1, dtype=torch.float32, device=self.dev)
                st.loss_host = torch.empty(1, dtype=torch.float32).pin_memory()
            st.s_out_host = torch.empty(T, self.C_s, dtype=dtype).pin_memory()
            st.sliced = [torch.cuda.Event() for _ in range(self.slices)]
            st.done = torch.cuda.Event()
            self.sets.append(st)
        self.key = (part.c.B, T, P)

    def _capture(self, k: int):
        # one eager pass first (launch attributes, tensor maps, the library's
        # own lazy set-up happen outside the capture)
        for idx in range(self.slices):
            self._piece(k, idx)
        torch.cuda.synchronize(self.dev)
        graphs = []
        for idx in range(self.slices):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._piece(k, idx)
            graphs.append(g)
        self.sets[k].graphs = graphs

    # -- steps ----------------------------------------------------------------------------
    def submit(self, lengths_host: torch.Tensor, s_host: torch.Tensor) -> int:
        """Enqueue one step: ``lengths_host`` (int32, B) and ``s_host`` (T x C_s),
        both in pinned host memory.  Returns a ticket for ``wait`` once the
        step's device work and read-backs are enqueued (after the partition's
        totals have come back, which also means the host inputs have been
        copied and may be reused)."""
        if lengths_host.dtype != torch.int32 or s_host.dim() != 2 or s_host.shape[1] != self.C_s:
            raise ValueError("lengths must be int32 (B,) and s (T, C_s)")
        main = torch.cuda.current_stream(self.dev)
        B, T = lengths_host.numel(), s_host.shape[0]
        self._ensure_inputs(B, T, s_host.dtype)
        ticket = self.submitted
        k = ticket % self.depth
        inp = self.inputs[k]
        # copies in and partition on the input stream, beside the running step
        with torch.cuda.stream(self.in_stream):
            if inp.used:
                self.in_stream.wait_event(inp.free)    # the slot's previous graphs have read them
            inp.lengths.copy_(lengths_host, non_blocking=True)
            inp.s.copy_(s_host, non_blocking=True)
            part = self._partition(inp, B, T, self.in_stream)
            inp.ready.record(self.in_stream)
        if self.key != (B, part.T, part.P):
            self._setup(part, s_host.dtype)           # drains: every slot's graphs are captured anew
        inp.part = part
        st = self.sets[k]
        if st.busy:
            main.wait_event(st.done)     # the slot's previous read-back has finished with z~ and s_out
        main.wait_event(inp.ready)
        if not st.graphs:
            self._capture(k)
        for idx in range(self.slices):
            st.graphs[idx].replay()
            st.sliced[idx].record(main)
        inp.free.record(main)
        inp.used = True
        with torch.cuda.stream(self.copy_stream):
            for idx in range(self.slices):
                c0, c1 = self.cuts[idx], self.cuts[idx + 1]
                self.copy_stream.wait_event(st.sliced[idx])
                if c1 > c0 and self.readback == "pair":
                    st.z_host[c0:c1].copy_(st.z[c0:c1], non_blocking=True)
            if self.readback == "loss":
                st.loss_host.copy_(st.loss, non_blocking=True)
            st.s_out_host.copy_(st.s_out, non_blocking=True)
            st.done.record(self.copy_stream)
        st.busy = True
        st.ticket = ticket
        self.submitted += 1
        return ticket

    def wait(self, ticket: int):
        """The pinned host results of step ``ticket``, valid until the step
        ``depth`` submissions later reuses them: (z~ of P x C_z, s_out of
        T x C_s) with readback "pair", (the Eq. 5 loss as a 1-element fp32
        tensor, s_out) with readback "loss"."""
        if self.sets and self.sets[ticket % self.depth].ticket == ticket:
            st = self.sets[ticket % self.depth]
        elif ticket in self.retired:
            st = self.retired.pop(ticket)
        else:
            raise ValueError(f"step {ticket} is no longer held (depth {self.depth})")
        st.done.synchronize()
        return (st.z_host if self.readback == "pair" else st.loss_host), st.s_out_host

    def run(self, lengths_host: torch.Tensor, s_host: torch.Tensor):
        """One step, waited for: returns the pinned host tensors of ``wait``,
        overwritten ``depth`` steps later."""
        return self.wait(self.submit(lengths_host, s_host))
