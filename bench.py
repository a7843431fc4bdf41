"""Benchmark of the packed single->pair->single block and varlen attention.

One step is one pass of the whole hot path:
  * the block on the near-uniform B=16 batch (N_i ~ U[700, 768], P =
    8,633,186 packed cells, C_s=384, C_z=128, transition 128->512->128, bf16
    I/O, fp32 accumulation), the largest single-GPU block workload:
    partition build + row splits, pair broadcast, transition, reduce + g;
  * varlen attention on the packed stream of 65,536 tokens (segments
    ~ U[16, 512], 12 heads x 64, bf16, non-causal).
``value`` is packed pair cells per second of the block (the block's P over
its device time per step); the attention's TFLOPS ride beside it in
``attn``.  L2 is flushed (a 512 MB write) before every timed step, outside
the timed events.  The partition build ends with a host readback; a short
device sleep after it (also outside the events) lets the host queue the
remaining calls ahead of the device, so each call's interval is device time.

The same line carries, measured in the same run: per-call figures of every
other block workload (``workloads``: the B=8 Pairformer batch, the
lognormal B=16 batch, the four stacked blocks of the skewed batch), the
packed-against-padded report (``packing``: cells, pair bytes, measured peak
allocation, block time) and the varlen-attention padding sweep
(``padsweep``).  ``--impl reference`` times the CPU oracle instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun every rank runs its own replica (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))
os.environ.setdefault("OMP_NUM_THREADS", str(os.cpu_count() or 1))

import numpy as np  # noqa: E402
import torch  # noqa: E402

from variable_length_batching_gb300 import workloads as wl  # noqa: E402

METRIC = "packed pair cells/sec per block and varlen attn TFLOPS; % of HBM/tensor roofline"
HOST_LEAD_CYCLES = 400_000     # ~0.2 ms of device sleep at 2 GHz, outside the timed intervals
BLOCK_CFG = wl.NEAR_UNIFORM_BF16          # the headline block workload
SIDE_BLOCK_CFGS = (wl.PAIRFORMER_BF16, wl.LOGNORMAL_BF16, wl.STACKED4_BF16)
ATTN_CFG = wl.VARLEN_ATTN_BF16
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20
L2_CLEAN_BYTES = 256 << 20
# kernels of ours launched per step: partition (scan and row splits in one
# launch), u/v projection, broadcast, transition, reduce, g projection,
# attention
LAUNCHES_PER_STEP = 7
SIDE_STEPS = 20                  # timed repetitions of each side report's calls
BACKWARD_CFG = wl.NEAR_UNIFORM_BF16  # the block backward on the headline batch
BACKWARD_STEPS = 3


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def traffic_record(kernel: str, workload: str):
    """Per-launch DRAM bytes of ``kernel`` on ``workload`` from a committed ncu
    capture, or None when there is none or the kernel's source changed
    since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("workload") != workload:
        return None
    src = os.path.join(ROOT, "variable_length_batching_gb300", "csrc", rec["source"])
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != rec["source_sha"]:
            return None
    return rec["bytes_per_launch"]


# ----------------------------------------------------------------------------
# Algorithmic work per call (what the method must do, not padded work)
# ----------------------------------------------------------------------------

def block_work(T, P, C_s, C_z, H_t, es=2):
    return {
        "partition": {"bytes": 0, "flops": 0},
        # the whole call (projection GEMM + broadcast): writes P*C_z outputs,
        # reads the singles and the two projection weights
        "broadcast": {"bytes": P * C_z * es + T * C_s * es + 2 * C_z * C_s * es,
                      "flops": 2 * 2 * T * C_s * C_z},
        # reads and writes every cell once; 2 GEMMs of C_z x H_t per cell
        "transition": {"bytes": 2 * P * C_z * es + 2 * H_t * C_z * es, "flops": 4 * C_z * H_t * P},
        # the whole call (reduce + g projection): reads every cell once;
        # writes m, reads s_in and W_g, writes s_out
        "reduce": {"bytes": P * C_z * es + T * C_z * es + 2 * T * C_s * es + C_s * C_z * es,
                   "flops": 2 * T * C_z * C_s},
    }


def attn_work(seqlens, H, d, es=2, causal=False):
    """QK^T and PV over the visible (query, key) pairs: n^2 per segment, or
    n (n + 1) / 2 under the causal mask; q, k, v read and o written once."""
    n = np.asarray(seqlens, dtype=np.int64)
    pairs = int((n * (n + 1) // 2).sum()) if causal else int((n * n).sum())
    return {"bytes": 4 * int(n.sum()) * H * d * es, "flops": 4 * pairs * H * d}


# ----------------------------------------------------------------------------
# Clock sampling during the timed region
# ----------------------------------------------------------------------------

_REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                "hw_thermal_slowdown": 0x40}


class _NvmlProbe:
    """SM clock, max SM clock and clock-event reasons of one GPU read through
    NVML (the library nvidia-smi reads), for sampling faster than nvidia-smi's
    loop.  Read-only queries."""

    def __init__(self, index):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        getter = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = getter or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def read(self):
        c = self.c
        clk, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if (self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(clk)) != 0 or      # 1 = NVML_CLOCK_SM
                self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, c.byref(mx)) != 0 or
                self.reasons_fn(self.h, c.byref(rs)) != 0):
            return None
        return float(clk.value), float(mx.value), int(rs.value)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """Clock and throttle-reason samples stamped on arrival: nvidia-smi's loop
    (every 20 ms) and, where libnvidia-ml loads, NVML reads every 2 ms, so that
    a timed region of a few tens of ms still holds samples.  Started before
    the warm-up; ``mark(start, end)`` is given the timed region's host clock
    (perf_counter) bounds, and the summary keeps only samples inside it."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20
    NVML_PERIOD_S = 0.002

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []          # (perf_counter, source, sm_mhz, max_mhz, set of reasons)
        self.window = None
        self.threads = []
        self.stop = None

    def _smi_reader(self, first):
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.proc.stdout:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            rs = {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}
            self.samples.append((time.perf_counter(), "nvidia-smi", sm, mx, rs))
            first.set()

    def _nvml_loop(self, probe):
        while not self.stop.is_set():
            r = probe.read()
            if r is not None:
                rs = {n for n, b in _REASON_BITS.items() if r[2] & b}
                self.samples.append((time.perf_counter(), "nvml", r[0], r[1], rs))
            self.stop.wait(self.NVML_PERIOD_S)
        probe.close()

    def __enter__(self):
        import threading
        self.stop = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.proc is not None:
            first = threading.Event()
            t = threading.Thread(target=self._smi_reader, args=(first,), daemon=True)
            t.start()
            self.threads.append(t)
            first.wait(timeout=10.0)        # sampling is running before any timed work
        try:
            probe = _NvmlProbe(self.gpu)
        except (OSError, AttributeError):
            probe = None
        if probe is not None:
            t = threading.Thread(target=self._nvml_loop, args=(probe,), daemon=True)
            t.start()
            self.threads.append(t)
        return self

    def mark(self, start, end):
        self.window = (start, end)

    def __exit__(self, *exc):
        self.stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
        for t in self.threads:
            t.join(timeout=5)

    def summary(self):
        lo, hi = self.window if self.window else (-float("inf"), float("inf"))
        inside = [s for s in list(self.samples) if lo <= s[0] <= hi]
        counts = {}
        for s in inside:
            counts[s[1]] = counts.get(s[1], 0) + 1
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": counts}
        reasons = set()
        for s in inside:
            reasons |= s[4]
        return {"sm_mhz": statistics.median(s[2] for s in inside), "sm_max_mhz": max(s[3] for s in inside),
                "sm_mhz_min": min(s[2] for s in inside), "reasons": sorted(reasons), "samples": counts}


# ----------------------------------------------------------------------------
# Multi-rank bookkeeping (replicas: no collective on the data path)
# ----------------------------------------------------------------------------

def max_over_ranks(values, world, device=None):
    """Element-wise max of per-rank timings (the job is as slow as its
    slowest rank); a no-op on one rank."""
    if world <= 1:
        return [float(v) for v in values]
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(units_per_rank, world, ms_max):
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time."""
    return world * units_per_rank / (ms_max * 1e-3)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def _dev_weights(w, dev):
    from types import SimpleNamespace
    g = lambda t: None if t is None else t.to(dev)
    return SimpleNamespace(W_a=g(w.W_a), W_b=g(w.W_b), ln_gamma=g(w.ln_gamma), ln_beta=g(w.ln_beta),
                           W1=g(w.W1), b1=g(w.b1), W2=g(w.W2), b2=g(w.b2), W_g=g(w.W_g), b_g=g(w.b_g))


class L2Flush:
    """Empties L2 between timed calls, outside their events: a write of a
    512 MB buffer, then a read of a 256 MB one (both larger than the 129 MB
    L2).  The read evicts the written lines, so their write-back to HBM
    happens here and not inside the next timed kernel."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=dev)

    def fill_(self, value):
        self.w.fill_(value)
        self.r.amax()


class BlockRun:
    """Device inputs and buffers of one block workload: the partition is
    built in every step; the pair state, the broadcast workspace and the
    singles outputs are allocated once.  A stacked workload chains its
    blocks through the singles, reusing one pair buffer."""

    def __init__(self, nt, cfg, dev, lengths=None):
        self.nt, self.cfg = nt, cfg
        self.inp = wl.make_block_inputs(cfg, lengths=lengths)
        self.ws = [_dev_weights(b, dev) for b in self.inp.blocks]
        self.lengths_d = torch.as_tensor(self.inp.lengths).to(dev)
        self.s_d = self.inp.s.to(dev)
        part = nt.nt_partition_build(self.lengths_d)
        self.T, self.P = part.T, part.P
        self.z = torch.empty(self.P, cfg.C_z, dtype=self.s_d.dtype, device=dev)
        self.wsp = torch.empty(max(nt.nt_pair_broadcast_workspace_bytes(self.T, cfg.C_z), 16), dtype=torch.uint8,
                               device=dev)
        self.m = torch.empty(self.T, cfg.C_z, dtype=self.s_d.dtype, device=dev)
        self.souts = [torch.empty_like(self.s_d) for _ in self.ws]

    @property
    def n_events(self):
        return 3 + 3 * len(self.ws)

    def step(self, ev, stream, attn=None):
        """One block step (and, with ``attn``, the attention call after it).
        ev[0..1] bracket the partition build (scan and row splits in one call,
        bounded by the singles' row count; it ends with the host reading the
        totals back); then per block k, ev[2+3k..5+3k] bracket its
        broadcast, transition and reduce; ev[-1] closes the attention call."""
        nt = self.nt
        ev[0].record(stream)
        p = nt.nt_partition_build(self.lengths_d, stream=stream, T=self.s_d.shape[0])
        ev[1].record(stream)
        # The partition's readback left the stream idle.  A short device
        # sleep, outside every timed interval, lets the host enqueue the next
        # calls ahead of the device, so their intervals hold device time and
        # not host launch latency.
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        ev[2].record(stream)
        s_cur = self.s_d
        for k, (w, so) in enumerate(zip(self.ws, self.souts)):
            nt.nt_pair_broadcast(p, s_cur, s_cur, w.W_a, w.W_b, z=self.z, workspace=self.wsp, stream=stream)
            ev[3 + 3 * k].record(stream)
            nt.nt_pair_transition(p, self.z, w.ln_gamma, w.ln_beta, w.W1, w.b1, w.W2, w.b2, out=self.z,
                                  stream=stream)
            ev[4 + 3 * k].record(stream)
            nt.nt_pair_reduce(p, self.z, w.W_g, w.b_g, s_in=s_cur, m=self.m, s_out=so, stream=stream)
            ev[5 + 3 * k].record(stream)
            s_cur = so
        if attn is not None:
            attn()
            ev[-1].record(stream)

    def call_times(self, evs):
        """Per-step ms of each call (summed over the stacked blocks)."""
        nb = len(self.ws)
        per = {"partition": [], "broadcast": [], "transition": [], "reduce": []}
        for ev in evs:
            per["partition"].append(ev[0].elapsed_time(ev[1]))
            for name, off in (("broadcast", 0), ("transition", 1), ("reduce", 2)):
                per[name].append(sum(ev[2 + 3 * k + off].elapsed_time(ev[3 + 3 * k + off]) for k in range(nb)))
        return per


def kstat(times_ms, w_bytes, w_flops, bound, peaks):
    """Achieved figure of one call against its bound, from its per-step
    times (mean; p10/p50/p90 beside it)."""
    ms = float(np.mean(times_ms))
    t = ms * 1e-3
    hbm, tc = peaks["hbm_gbs"], peaks["bf16_tflops"]
    spread = {"ms": ms, "ms_p10_p50_p90": [float(x) for x in np.percentile(times_ms, [10, 50, 90])]}
    if bound == "tensor":
        a = w_flops / t / 1e12
        out = {"bound": "tensor", "achieved": a, "peak": tc, "unit": "TFLOP/s", "frac": a / tc}
        # attainable roofline: min(tensor peak, arithmetic intensity x HBM bandwidth)
        att = min(tc, w_flops / w_bytes * hbm / 1e3)
        out.update({"attainable": att, "frac_attainable": a / att})
    else:
        a = w_bytes / t / 1e9
        out = {"bound": "hbm", "achieved": a, "peak": hbm, "unit": "GB/s", "frac": a / hbm}
    out.update(spread)
    return out


def block_kernels(run, per, peaks):
    """Per-call roofline figures of one block workload: broadcast and reduce
    are whole calls (projection GEMM included), against HBM; the transition
    against the bf16 tensor peak.  Work and times are summed over stacked
    blocks."""
    cfg, nb = run.cfg, len(run.ws)
    es = 2 if cfg.dtype == wl.BF16 else 4
    work = block_work(run.T, run.P, cfg.C_s, cfg.C_z, cfg.H_t, es)
    return {
        "broadcast": dict(kstat(per["broadcast"], nb * work["broadcast"]["bytes"], 0, "hbm", peaks),
                          call="whole call: u/v projection GEMM + broadcast kernel"),
        "transition": kstat(per["transition"], nb * work["transition"]["bytes"], nb * work["transition"]["flops"],
                            "tensor", peaks),
        "reduce": dict(kstat(per["reduce"], nb * work["reduce"]["bytes"], 0, "hbm", peaks),
                       call="whole call: reduce kernel + g projection GEMM"),
        "partition": {"ms": float(np.mean(per["partition"])), "note": "scan + row splits + one totals readback"},
    }


def run_gpu(args, rank, world, local_rank):
    from variable_length_batching_gb300 import build, nt
    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()

    # ---- inputs, resident in HBM before the timed region ----
    run = BlockRun(nt, BLOCK_CFG, dev)
    ainp = wl.make_attn_inputs(ATTN_CFG)
    apart = nt.nt_partition_build(torch.as_tensor(ainp.seqlens).to(dev))   # cu_seqlens on the device
    cu_d = apart.cu_seqlens
    q_d, k_d, v_d = ainp.q.to(dev), ainp.k.to(dev), ainp.v.to(dev)
    max_len = apart.max_len
    o_d = torch.empty_like(q_d)
    attn_ws = torch.empty(nt.nt_varlen_attn_workspace_bytes(), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    T, P = run.T, run.P
    C_s, C_z, H_t = BLOCK_CFG.C_s, BLOCK_CFG.C_z, BLOCK_CFG.H_t

    attn = lambda: nt.nt_varlen_attn(q_d, k_d, v_d, cu_d, max_len, out=o_d, stream=stream, workspace=attn_ws)

    def new_events(n):
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    for _ in range(args.warmup):
        flush.fill_(1.0)
        run.step(new_events(run.n_events + 1), stream, attn)
    nt.nt_device_status(stream)

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    evs = []
    with ClockSampler(local_rank) as clk:
        t0 = time.perf_counter()
        for _ in range(args.steps):
            flush.fill_(float(len(evs)))     # L2 flush, outside the step's events
            ev = new_events(run.n_events + 1)
            run.step(ev, stream, attn)
            evs.append(ev)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        wall = t1 - t0
        clk.mark(t0, t1)
    if world > 1:
        dist.barrier()
    nt.nt_device_status(stream)

    per = run.call_times(evs)
    per["attention"] = [ev[-2].elapsed_time(ev[-1]) for ev in evs]
    ms = {n: float(np.mean(v)) for n, v in per.items()}
    block_ms = ms["partition"] + ms["broadcast"] + ms["transition"] + ms["reduce"]
    step_ms = block_ms + ms["attention"]
    block_ms_max, attn_ms_max, step_ms_max = max_over_ranks([block_ms, ms["attention"], step_ms], world, dev)

    # ---- end to end through the C ABI with host buffers ----
    e2e = run_e2e(nt, run.inp, dev, stream, args)

    # ---- the other block workloads, packing and padding reports (same run) ----
    side_steps = max(3, min(args.steps, SIDE_STEPS))
    workloads = {BLOCK_CFG.name: None}
    for cfg in SIDE_BLOCK_CFGS:
        workloads[cfg.name] = measure_block(nt, cfg, dev, stream, flush, side_steps, args.warmup, peaks)
    del run.z
    torch.cuda.empty_cache()
    packing = run_packing(nt, dev, stream, flush, side_steps)
    padsweep = run_padsweep(nt, dev, stream, flush, side_steps, peaks)
    backward = {"attention": measure_attn_backward(nt, dev, stream, flush, side_steps, peaks, ainp, q_d, k_d, v_d,
                                                   cu_d, max_len),
                "block": measure_block_backward(nt, BACKWARD_CFG, dev, stream, flush, BACKWARD_STEPS, peaks)}

    if rank != 0:
        return None
    aw = attn_work(ainp.seqlens, ATTN_CFG.H, ATTN_CFG.d)
    kernels = block_kernels(run, per, peaks)
    kernels["attention"] = kstat(per["attention"], aw["bytes"], aw["flops"], "tensor", peaks)
    workloads[BLOCK_CFG.name] = {"B": BLOCK_CFG.B, "T": T, "P": P, "blocks": 1, "block_ms": block_ms,
                                 "cells_per_s": P / (block_ms * 1e-3), "steps": args.steps,
                                 "kernels": {k: v for k, v in kernels.items() if k != "attention"},
                                 "note": "the headline workload (the main timed steps)"}
    # the kernel with the largest share of the step's device time
    dom = max(("broadcast", "transition", "reduce", "attention"), key=lambda n: ms[n])
    roof = {k: v for k, v in kernels[dom].items() if not k.startswith("ms") and k != "call"}
    roof["kernel"] = dom
    roof["share_of_step"] = ms[dom] / step_ms
    roof["peak_source"] = f"{peak_src} ({'burst copy' if roof['bound'] == 'hbm' else 'cuBLAS bf16 burst'})"
    roof["traffic"] = traffic_record(dom, BLOCK_CFG.name if dom != "attention" else ATTN_CFG.name)
    cells_per_s = job_throughput(P, world, block_ms_max)
    attn_tflops = job_throughput(aw["flops"], world, attn_ms_max) / 1e12
    nmax = int(run.inp.lengths.max())
    line = {
        "metric": METRIC,
        "value": cells_per_s,
        "unit": "pair cells/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded numpy draws of the pages' workload shapes; random-init weights)",
        "config": {"workload": f"block: {BLOCK_CFG.name} (T={T}, P={P} packed cells vs "
                               f"{BLOCK_CFG.B * nmax ** 2} padded); "
                               f"attention: {ATTN_CFG.name} ({len(ainp.seqlens)} segments)",
                   "B": BLOCK_CFG.B, "T": T, "P": P, "C_s": C_s, "C_z": C_z, "H_t": H_t,
                   "attn_T": int(ainp.seqlens.sum()), "attn_segments": int(len(ainp.seqlens)),
                   "heads": ATTN_CFG.H, "head_dim": ATTN_CFG.d,
                   "l2": "flushed before every timed step, outside the events: a 512 MB write, then a 256 MB "
                         "read so that the write's dirty lines are written back before the step",
                   "parallelism": f"replicas x{world}"},
        "block_ms": block_ms_max,
        "attn": {"tflops": attn_tflops, "ms": attn_ms_max, "flops_per_step": aw["flops"],
                 "roofline": {k: v for k, v in kernels["attention"].items() if not k.startswith("ms")}},
        "kernels": kernels,
        "roofline": roof,
        "workloads": workloads,
        "packing": packing,
        "padsweep": padsweep,
        "backward": backward,
        "e2e": e2e,
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
    }
    return line


def _event_ms(fn, stream, flush, steps, warmup=3):
    """Mean CUDA-event time (ms) of ``fn`` on ``stream``, L2 flushed before each run."""
    for _ in range(warmup):
        flush.fill_(0.0)
        fn()
    times = []
    for i in range(steps):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in times]))


def fp32_fma_tflops(dev, peaks):
    """fp32 FMA peak: 128 lanes per SM per clock x 2 flop x SMs x max SM clock."""
    mhz = peaks.get("sm_max_mhz", 2070.0)
    return 2 * 128 * torch.cuda.get_device_properties(dev).multi_processor_count * mhz * 1e6 / 1e12


def measure_attn_backward(nt, dev, stream, flush, steps, peaks, ainp, q, k, v, cu, max_len):
    """dq, dk, dv of the attention stream for a seeded upstream gradient
    (the forward's o and lse made once, outside the timed calls)."""
    o = torch.empty_like(q)
    _, lse = nt.nt_varlen_attn_qk(q, k, v, cu, cu, max_len, out=o, want_lse=True, stream=stream)
    d_o = wl.random_rows(q.shape[0] * ATTN_CFG.H, ATTN_CFG.d, ATTN_CFG.dtype, seed=1).reshape(q.shape).to(dev)
    ms = _event_ms(lambda: nt.nt_varlen_attn_bwd(q, k, v, o, d_o, lse, cu, None, max_len, stream=stream),
                   stream, flush, steps)
    nt.nt_device_status(stream)
    aw = attn_work(ainp.seqlens, ATTN_CFG.H, ATTN_CFG.d)
    flops = 2.5 * aw["flops"]        # S recomputed, dV, dP, dQ, dK: 2.5 times the forward's flops
    return {"workload": ATTN_CFG.name, "ms": ms, "bound": "tensor", "achieved": flops / ms / 1e9,
            "unit": "TFLOP/s", "peak": peaks["bf16_tflops"], "frac": flops / ms / 1e9 / peaks["bf16_tflops"],
            "flops": flops, "steps": steps, "call": "dQ kernel (forms D) + dK/dV kernel"}


def backward_route(cfg):
    """The pair-cell part of the block backward runs on the tensor cores for
    bf16 with C_z = 128 and H_t a multiple of 128, else on CUDA cores."""
    return "tensor" if cfg.dtype == wl.BF16 and cfg.C_z == 128 and cfg.H_t % 128 == 0 else "fma"


def backward_roof(route, flops, ms, dev, peaks):
    """Achieved algorithmic TFLOP/s against the bf16 tensor peak (tensor-core
    route) or the derived fp32 FMA peak (CUDA-core route)."""
    achieved = flops / ms / 1e9
    if route == "tensor":
        return {"bound": "tensor", "achieved": achieved, "unit": "TFLOP/s", "peak": peaks["bf16_tflops"],
                "frac": achieved / peaks["bf16_tflops"], "peak_source": "measured bf16"}
    peak = fp32_fma_tflops(dev, peaks)
    return {"bound": "alu", "achieved": achieved, "unit": "TFLOP/s", "peak": peak, "frac": achieved / peak,
            "peak_source": "fp32 FMA: 128 lanes per SM per clock x 2 flop x SMs x max SM clock"}


def measure_block_backward(nt, cfg, dev, stream, flush, steps, peaks):
    """The Eq. 5 loss and the block's gradients on one block workload; the
    forward's outputs are made once, outside the timed calls."""
    inp = wl.make_block_inputs(cfg)
    wd = _dev_weights(inp.blocks[0], dev)
    s = inp.s.to(dev)
    part = nt.nt_partition_build(torch.as_tensor(inp.lengths).to(dev))
    z, m, s_out = nt.block_forward(part, s, wd, stream=stream)
    dt = nt._dtype(s)
    ws = torch.empty(nt.nt_pair_block_loss_backward_workspace_bytes(dt, part.T, part.P, cfg.C_s, cfg.C_z, cfg.H_t),
                     dtype=torch.uint8, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)

    def fused():
        nt.nt_pair_block_loss_backward(part, s, wd, m, s_out, z, loss=loss, workspace=ws, stream=stream)
    ms = _event_ms(fused, stream, flush, steps, warmup=2)
    del ws
    ws2 = torch.empty(nt.nt_pair_block_backward_workspace_bytes(dt, part.T, part.P, cfg.C_z, cfg.H_t),
                      dtype=torch.uint8, device=dev)

    def two_calls():
        _, ds_out, dz = nt.nt_pair_block_loss(part, s_out, z, stream=stream)
        nt.nt_pair_block_backward(part, s, wd, m, ds_out, dz, workspace=ws2, stream=stream)
    ms2 = _event_ms(two_calls, stream, flush, steps, warmup=2)
    nt.nt_device_status(stream)
    # per cell: A recomputed, dH, dY, dW1, dW2 (five C_z x H_t products)
    flops = 5 * 2 * cfg.C_z * cfg.H_t * part.P
    route = backward_route(cfg)
    out = {"workload": cfg.name, "P": part.P, "ms": ms, "flops": flops, "steps": steps,
           **backward_roof(route, flops, ms, dev, peaks),
           "call": "nt_pair_block_loss_backward ("
                   + ("pair cells on tcgen05 GEMMs" if route == "tensor" else "fp32 CUDA cores") + ")",
           "two_calls_ms": ms2}
    del z, m, s_out, ws2
    torch.cuda.empty_cache()
    return out


def measure_block(nt, cfg, dev, stream, flush, steps, warmup, peaks):
    """Per-call figures of one block workload: ``steps`` block steps with L2
    flushed before each, per-call CUDA events."""
    run = BlockRun(nt, cfg, dev)
    for _ in range(max(3, warmup)):
        flush.fill_(0.0)
        run.step([torch.cuda.Event(enable_timing=True) for _ in range(run.n_events)], stream)
    evs = []
    for i in range(steps):
        flush.fill_(float(i))
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(run.n_events)]
        run.step(ev, stream)
        evs.append(ev)
    torch.cuda.synchronize()
    nt.nt_device_status(stream)
    per = run.call_times(evs)
    ms = {n: float(np.mean(v)) for n, v in per.items()}
    block_ms = sum(ms.values())
    nb = len(run.ws)
    out = {"B": cfg.B, "T": run.T, "P": run.P, "blocks": nb, "block_ms": block_ms,
           "cells_per_s": nb * run.P / (block_ms * 1e-3), "steps": steps,
           "kernels": block_kernels(run, per, peaks),
           "graph": measure_block_graph(nt, run, stream, flush, steps)}
    del run
    torch.cuda.empty_cache()
    return out


def measure_block_graph(nt, run, stream, flush, steps):
    """The block's calls (every stacked block's broadcast, transition and
    reduce) captured once in a CUDA graph over a partition built beforehand,
    and timed per replay with L2 flushed before each: the device time of the
    calls with no host launch gaps between them (the partition build, which
    reads its totals back to the host, is outside)."""
    part = nt.nt_partition_build(run.lengths_d, T=run.s_d.shape[0])

    def calls():
        s_cur = run.s_d
        for w, so in zip(run.ws, run.souts):
            nt.nt_pair_broadcast(part, s_cur, s_cur, w.W_a, w.W_b, z=run.z, workspace=run.wsp)
            nt.nt_pair_transition(part, run.z, w.ln_gamma, w.ln_beta, w.W1, w.b1, w.W2, w.b2, out=run.z)
            nt.nt_pair_reduce(part, run.z, w.W_g, w.b_g, s_in=s_cur, m=run.m, s_out=so)
            s_cur = so

    with torch.cuda.stream(stream):
        calls()                                   # lazy set-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls()
        for i in range(3):
            flush.fill_(float(i))
            g.replay()
        times = []
        for i in range(steps):
            flush.fill_(float(i))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize()
    nt.nt_device_status(stream)
    t = [a.elapsed_time(b) for a, b in times]
    ms = float(np.mean(t))
    del g
    return {"block_ms": ms, "ms_p10_p50_p90": [float(x) for x in np.percentile(t, [10, 50, 90])],
            "cells_per_s": len(run.ws) * run.P / (ms * 1e-3),
            "note": "broadcast, transition and reduce replayed as one CUDA graph; partition built beforehand"}


def run_e2e(nt, binp, dev, stream, args):
    """The block host to host through the package's BlockGraph.  Every step
    copies the lengths and the singles in from pinned host memory, rebuilds
    the partition (a totals read-back), replays the captured broadcast ->
    transition -> reduce graph, computes the Eq. 5 loss of the step's two
    outputs on the device and reads the loss and s_out back.  Two steps are
    in flight: step i is submitted before step i - 1's results are waited
    for, so its copies in, partition and compute overlap the previous
    step's read-back.  The timed region ends once the last step's results
    are on the host.  The block's weights are resident on the device, as a
    model's parameters are.  ``pair_readback`` measures the same steps
    reading the whole pair output z~ back instead of the loss (three
    transition slices, each read back on a second stream as soon as it is
    done), which the host link bounds."""
    from variable_length_batching_gb300 import graph
    host = {"lengths": torch.as_tensor(binp.lengths).pin_memory(), "s": binp.s.pin_memory()}
    T = int(binp.lengths.sum())
    P = int((binp.lengths.astype(np.int64) ** 2).sum())
    h2d = sum(t.numel() * t.element_size() for t in host.values())

    def measure(readback):
        runner = graph.BlockGraph(_dev_weights(binp.blocks[0], dev), depth=2, readback=readback)

        def steps(n, pipelined):
            tickets = []
            for i in range(n):
                tickets.append(runner.submit(host["lengths"], host["s"]))
                if not pipelined:
                    runner.wait(tickets[i])
                elif i >= 1:
                    runner.wait(tickets[i - 1])
            if pipelined and tickets:
                runner.wait(tickets[-1])

        def timed(pipelined):
            steps(max(args.warmup, 3), pipelined)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            steps(args.steps, pipelined)
            torch.cuda.synchronize()
            return (time.perf_counter() - t0) / args.steps

        dt_seq = timed(False)
        dt = timed(True)
        out_bytes = (P * BLOCK_CFG.C_z * 2 if readback == "pair" else 4) + T * BLOCK_CFG.C_s * 2
        path = ("pinned host -> H2D of lengths and singles -> nt_partition_build (totals read-back) -> "
                + (f"CUDA-graph replays of broadcast / transition in {runner.slices} slices growing "
                   f"x{runner.growth:g} / reduce, with each slice's z~ and then s_out read back on a second stream"
                   if readback == "pair" else
                   "one CUDA-graph replay of broadcast / transition / reduce / Eq. 5 loss, then the loss and "
                   "s_out read back on a second stream")
                + f"; {runner.depth} steps in flight (weights resident on the device)")
        res = {"value": P / dt, "unit": "pair cells/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(out_bytes + 4 * 8),   # + the partition's four totals
               "ms_per_step": dt * 1e3, "ms_per_step_one_at_a_time": dt_seq * 1e3, "path": path}
        del runner
        torch.cuda.empty_cache()
        return res

    e2e = measure("loss")
    e2e["pair_readback"] = measure("pair")
    return e2e


# ----------------------------------------------------------------------------
# CPU oracle: the baseline beside the GPU number, and the reference arm
# ----------------------------------------------------------------------------

class OracleBlock:
    """The oracle on the headline block workload, one sample at a time (its
    own loop is per sample, so a sample is the natural bounded unit)."""

    def __init__(self):
        from oracle import block as oblock
        self.ob = oblock
        binp = wl.make_block_inputs(BLOCK_CFG)
        w = binp.blocks[0]
        f = wl.io_bits_to_f64
        self.w = oblock.Weights(f(w.W_a), f(w.W_b), f(w.ln_gamma), f(w.ln_beta), 1e-5, f(w.W1), None, f(w.W2),
                                None, f(w.W_g), None)
        self.lengths = binp.lengths
        self.cu = np.concatenate([[0], np.cumsum(binp.lengths.astype(np.int64))])
        self.s = f(binp.s)

    def sample(self, b):
        """Runs sample b of the batch; returns its pair cells."""
        n = int(self.lengths[b])
        self.ob.block_packed(self.lengths[b:b + 1], self.s[self.cu[b]:self.cu[b] + n], self.w)
        return n * n


def oracle_block_sample(budget_s=12.0):
    """The oracle on the headline block workload, whole samples in batch
    order until ``budget_s`` of CPU time has passed; returns (cells/s, what
    the sample was)."""
    ob = OracleBlock()
    cells, b, t0 = 0, 0, time.perf_counter()
    while True:
        cells += ob.sample(b % BLOCK_CFG.B)
        b += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return cells / dt, (f"the first {b} of the {BLOCK_CFG.B} samples of the near-uniform batch "
                        f"({cells} pair cells, every step of the block per sample), {dt:.1f} s")


def oracle_attn_sample(budget_s=8.0):
    from oracle import attention as oattn
    a = wl.make_attn_inputs(ATTN_CFG)
    f = wl.io_bits_to_f64
    q, k, v = f(a.q), f(a.k), f(a.v)
    from oracle.partition import partition
    cu = partition(a.seqlens).cu_seqlens
    flops, t0, seg = 0, time.perf_counter(), 0
    while time.perf_counter() - t0 < budget_s and seg < len(a.seqlens):
        oattn.varlen_attention(q, k, v, cu, segments=[seg])
        flops += 4 * int(a.seqlens[seg]) ** 2 * ATTN_CFG.H * ATTN_CFG.d
        seg += 1
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, f"first {seg} of {len(a.seqlens)} segments, {dt:.1f} s"


def cpu_cores():
    return os.cpu_count() or 1


def cpu_threads():
    """Thread counts in effect for the oracle's numpy/BLAS calls: bench.py
    sets both variables to the core count before numpy loads, unless the
    caller set them."""
    return {"OPENBLAS_NUM_THREADS": int(os.environ.get("OPENBLAS_NUM_THREADS", "1")),
            "OMP_NUM_THREADS": int(os.environ.get("OMP_NUM_THREADS", "1"))}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on the headline workload: each
    step runs one whole sample of the near-uniform batch (samples in batch
    order, about 1.5 s each on 16 cores); value = pair cells per second."""
    if rank != 0:
        return None
    ob = OracleBlock()
    for i in range(min(args.warmup, 1)):
        ob.sample(i)
    cells, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        cells += ob.sample(i % BLOCK_CFG.B)
    wall = time.perf_counter() - t0
    value = cells / wall
    sample = (f"{args.steps} steps, one whole sample of the near-uniform batch per step ({cells} pair cells), "
              f"{wall:.1f} s")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "pair cells/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * wall / max(args.steps, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded numpy draws of the pages' workload shapes; random-init weights)",
        "config": {"workload": f"block: {BLOCK_CFG.name} (CPU oracle, float64, one sample per step)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "pair cells/s", "cores": cpu_cores(), "threads": cpu_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "pair cells/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }


WORKLOADS = {"pairformer": wl.PAIRFORMER_BF16, "lognormal": wl.LOGNORMAL_BF16,
             "near_uniform": wl.NEAR_UNIFORM_BF16, "stacked4": wl.STACKED4_BF16, "tiny": wl.TINY_FP32}


def _timed(fn, flush, reps, stream):
    """Median, p10 and p90 (ms) of ``reps`` runs of ``fn`` with L2 flushed before each."""
    ts = []
    for i in range(reps):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    v = [a.elapsed_time(b) for a, b in ts]
    return [float(x) for x in np.percentile(v, [50, 10, 90])]


def run_packing(nt, dev, stream, flush, steps):
    """Packed against padded pair state for every block workload: cells and
    bytes of the pair tensor, measured peak device allocation of one block
    (all four chained blocks for the stacked workload, with the pair buffer
    reused and with every block's pair output retained), and block time.  The
    padded rows run the same kernels on every sample padded to N_max, the
    cost a padded layout pays.  Returns one record per workload."""
    out = []
    for name in ("tiny", "pairformer", "lognormal", "near_uniform", "stacked4"):
        cfg = WORKLOADS[name]
        base = wl.make_block_inputs(cfg)
        nmax = int(base.lengths.max())
        es = 2 if cfg.dtype == wl.BF16 else 4
        line = {"workload": cfg.name, "B": cfg.B, "C_z": cfg.C_z, "blocks": cfg.n_blocks,
                "lengths": [int(x) for x in base.lengths]}
        for layout, lens in (("packed", base.lengths), ("padded", np.full(cfg.B, nmax, dtype=np.int32))):
            inp = wl.make_block_inputs(cfg, lengths=lens)
            ws = [_dev_weights(b, dev) for b in inp.blocks]
            lengths_d = torch.as_tensor(inp.lengths).to(dev)
            s0 = inp.s.to(dev)
            torch.cuda.synchronize()
            res = {}
            for mode in (("reuse", "retain") if cfg.n_blocks > 1 else ("reuse",)):
                torch.cuda.synchronize()
                torch.cuda.reset_peak_memory_stats(dev)
                before = torch.cuda.memory_allocated(dev)
                keep = []
                part = nt.nt_partition_build(lengths_d)
                s_cur, z = s0, None
                for w in ws:
                    z_k, _, s_cur = nt.block_forward(part, s_cur, w, z=None if mode == "retain" else z)
                    z = z_k
                    if mode == "retain":
                        keep.append(z_k)
                torch.cuda.synchronize()
                res[mode] = torch.cuda.max_memory_allocated(dev) - before
                del keep, z, z_k, s_cur, part
            part = nt.nt_partition_build(lengths_d)
            z = torch.empty(part.P, cfg.C_z, dtype=s0.dtype, device=dev)
            wsp = torch.empty(nt.nt_pair_broadcast_workspace_bytes(part.T, cfg.C_z), dtype=torch.uint8, device=dev)
            sos = [torch.empty_like(s0) for _ in ws]
            m = torch.empty(part.T, cfg.C_z, dtype=s0.dtype, device=dev)

            def chain():
                s_cur = s0
                for w, so in zip(ws, sos):
                    nt.nt_pair_broadcast(part, s_cur, s_cur, w.W_a, w.W_b, z=z, workspace=wsp, stream=stream)
                    nt.nt_pair_transition(part, z, w.ln_gamma, w.ln_beta, w.W1, w.b1, w.W2, w.b2, out=z,
                                          stream=stream)
                    nt.nt_pair_reduce(part, z, w.W_g, w.b_g, s_in=s_cur, m=m, s_out=so, stream=stream)
                    s_cur = so
            for _ in range(3):
                chain()
            med, p10, p90 = _timed(chain, flush, steps, stream)
            line[layout] = {"cells": int(part.P), "pair_bytes": int(part.P) * cfg.C_z * es,
                            "peak_alloc_bytes": res, "ms": med, "ms_p10_p90": [p10, p90],
                            "cells_per_s": part.P * cfg.n_blocks / (med * 1e-3)}
            del z, wsp, sos, m, part, ws, s0
            torch.cuda.empty_cache()
        line["pair_bytes_ratio"] = line["padded"]["pair_bytes"] / line["packed"]["pair_bytes"]
        line["peak_alloc_ratio"] = line["padded"]["peak_alloc_bytes"]["reuse"] / line["packed"]["peak_alloc_bytes"]["reuse"]
        line["speedup_packed_over_padded"] = line["padded"]["ms"] / line["packed"]["ms"]
        out.append(line)
    nt.nt_device_status(stream)
    return out


def _device_qkv(T, H, d, seed, dev):
    """N(0, 1) q, k, v of T tokens drawn on the device from a seeded
    generator (timing inputs of the padding sweep, where the host draw of
    the padded layouts would take longer than the measurement)."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    return [torch.randn(T, H, d, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
            for _ in range(3)]


def run_padsweep(nt, dev, stream, flush, steps, peaks):
    """Varlen attention over the packed stream against the same kernel on the
    same number of segments padded to 512 tokens, at equivalent padding rates
    from 3% to 90% (65,536 real tokens, 12 heads x 64).  Returns one record
    per rate."""
    out = []
    ws = torch.empty(nt.nt_varlen_attn_workspace_bytes(), dtype=torch.uint8, device=dev)
    for rate in wl.PADDING_SWEEP:
        lo, hi = wl.sweep_length_range(rate)
        rng = np.random.default_rng(0)
        lens = wl.draw_segments(ATTN_CFG.total_tokens, lo, hi, rng)
        line = {"target_rate": rate, "len_range": [lo, hi], "segments": int(len(lens)), "pad_to": wl.PAD_TO,
                "equivalent_pad_rate": 1.0 - float(lens.sum()) / (len(lens) * wl.PAD_TO)}
        w = attn_work(lens, ATTN_CFG.H, ATTN_CFG.d)
        for layout, L in (("varlen", lens), ("padded", np.full(len(lens), wl.PAD_TO, dtype=np.int32))):
            part = nt.nt_partition_build(torch.as_tensor(L).to(dev))
            q, k, v = _device_qkv(int(L.sum()), ATTN_CFG.H, ATTN_CFG.d, 0, dev)
            o = torch.empty_like(q)
            fn = lambda: nt.nt_varlen_attn(q, k, v, part.cu_seqlens, part.max_len, out=o, stream=stream,
                                           workspace=ws)
            for _ in range(3):
                fn()
            med, p10, p90 = _timed(fn, flush, steps, stream)
            line[layout] = {"tokens": int(L.sum()), "ms": med, "ms_p10_p90": [p10, p90],
                            "useful_tflops": w["flops"] / (med * 1e-3) / 1e12}
            del q, k, v, o, part
            torch.cuda.empty_cache()
        line["measured_savings"] = 1.0 - line["varlen"]["ms"] / line["padded"]["ms"]
        line["varlen_frac_of_peak"] = line["varlen"]["useful_tflops"] / peaks["bf16_tflops"]
        out.append(line)
    nt.nt_device_status(stream)
    return out


def _report_setup():
    from variable_length_batching_gb300 import build, nt
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    return nt, dev, stream, flush


def run_rect(args):
    """The rectangular block (N_i x M_i pair states, distinct row and column
    singles) on the B=8 batch with N_i, M_i ~ U[64, 256]: per-call device
    time (L2 flushed), cells/s of the block and the broadcast/reduce HBM
    fractions.  One JSON line."""
    from variable_length_batching_gb300 import build, nt
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    peaks, _ = load_peaks()
    cfg = wl.RECT_BF16
    inp = wl.make_rect_inputs(cfg)
    w = _dev_weights(inp.blocks[0], dev)
    part = nt.nt_partition_build_rect(torch.as_tensor(inp.rows).to(dev), torch.as_tensor(inp.cols).to(dev))
    sr, sc = inp.s_row.to(dev), inp.s_col.to(dev)
    z = torch.empty(part.P, cfg.C_z, dtype=sr.dtype, device=dev)
    ws = torch.empty(nt.nt_pair_broadcast_workspace_bytes_rect(part.T, part.T_cols, cfg.C_z), dtype=torch.uint8,
                     device=dev)
    m = torch.empty(part.T, cfg.C_z, dtype=sr.dtype, device=dev)
    so = torch.empty_like(sr)
    calls = {
        "broadcast": lambda: nt.nt_pair_broadcast(part, sr, sc, w.W_a, w.W_b, z=z, workspace=ws, stream=stream),
        "transition": lambda: nt.nt_pair_transition(part, z, w.ln_gamma, w.ln_beta, w.W1, w.b1, w.W2, w.b2,
                                                    out=z, stream=stream),
        "reduce": lambda: nt.nt_pair_reduce(part, z, w.W_g, w.b_g, s_in=sr, m=m, s_out=so, stream=stream),
    }
    for _ in range(3):
        for f in calls.values():
            f()
    out = {"report": "rect", "workload": cfg.name, "T_rows": part.T, "T_cols": part.T_cols, "P": part.P}
    tot = 0.0
    for name, f in calls.items():
        med, p10, p90 = _timed(f, flush, args.steps, stream)
        out[name] = {"ms": med, "ms_p10_p90": [p10, p90]}
        tot += med
    es = 2
    out["broadcast"]["hbm_frac"] = part.P * cfg.C_z * es / (out["broadcast"]["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]
    out["reduce"]["hbm_frac"] = part.P * cfg.C_z * es / (out["reduce"]["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]
    out["transition"]["tensor_frac"] = (4 * cfg.C_z * cfg.H_t * part.P / (out["transition"]["ms"] * 1e-3) / 1e12
                                        / peaks["bf16_tflops"])
    out["block_ms"] = tot
    out["cells_per_s"] = part.P / (tot * 1e-3)
    nt.nt_device_status(stream)
    print(json.dumps(out), flush=True)


def run_only(args):
    """Time one call on one workload (profiling and per-kernel rooflines):
    ``--only {partition,broadcast,transition,reduce,block,attention}``."""
    from variable_length_batching_gb300 import build, nt
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()
    flush = L2Flush(dev)
    if args.only == "attention":
        cfg = ATTN_CFG
        a = wl.make_attn_inputs(cfg)
        apart = nt.nt_partition_build(torch.as_tensor(a.seqlens).to(dev))
        cu, ml = apart.cu_seqlens, apart.max_len
        q, k, v = a.q.to(dev), a.k.to(dev), a.v.to(dev)
        o = torch.empty_like(q)
        aws = torch.empty(nt.nt_varlen_attn_workspace_bytes(), dtype=torch.uint8, device=dev)
        if args.causal:
            fn = lambda: nt.nt_varlen_attn_qk(q, k, v, cu, cu, ml, causal=True, out=o, stream=stream, workspace=aws)
        else:
            fn = lambda: nt.nt_varlen_attn(q, k, v, cu, ml, out=o, stream=stream, workspace=aws)
        w = attn_work(a.seqlens, cfg.H, cfg.d, causal=args.causal)
        bound, name = "tensor", cfg.name + ("_causal" if args.causal else "")
        if args.backward:
            # the forward's o and lse, then dq, dk, dv for a seeded upstream gradient
            _, lse_f = nt.nt_varlen_attn_qk(q, k, v, cu, cu, ml, causal=args.causal, out=o, want_lse=True)
            do = wl.random_rows(q.shape[0] * cfg.H, cfg.d, cfg.dtype, seed=1).reshape(q.shape).to(dev)
            fn = lambda: nt.nt_varlen_attn_bwd(q, k, v, o, do, lse_f, cu, None, ml, causal=args.causal,
                                               stream=stream)
            # S recomputed, dV, dP, dQ, dK: 2.5 times the forward's flops; q, k, v, o, dO read,
            # dq, dk, dv written
            w = {"flops": int(2.5 * w["flops"]), "bytes": 2 * w["bytes"]}
            name += "_backward"
    else:
        cfg = WORKLOADS[args.workload]
        inp = wl.make_block_inputs(cfg)
        wd = _dev_weights(inp.blocks[0], dev)
        lengths = torch.as_tensor(inp.lengths).to(dev)
        s = inp.s.to(dev)
        part = nt.nt_partition_build(lengths)
        z = nt.nt_pair_broadcast(part, s, s, wd.W_a, wd.W_b)
        ws = torch.empty(nt.nt_pair_broadcast_workspace_bytes(part.T, cfg.C_z), dtype=torch.uint8, device=dev)
        wsf = torch.empty(nt.lib().nt_pair_block_fused_workspace_bytes(part.T, part.T, cfg.C_z), dtype=torch.uint8,
                          device=dev)
        zt = torch.empty_like(z)
        m = torch.empty(part.T, cfg.C_z, dtype=z.dtype, device=dev)
        so = torch.empty(part.T, cfg.C_s, dtype=z.dtype, device=dev)
        es = 2 if cfg.dtype == wl.BF16 else 4
        bw = block_work(part.T, part.P, cfg.C_s, cfg.C_z, cfg.H_t, es)
        fns = {
            "partition": (lambda: nt.nt_partition_build(lengths, stream=stream, T=s.shape[0]), bw["partition"],
                          "latency"),
            "broadcast": (lambda: nt.nt_pair_broadcast(part, s, s, wd.W_a, wd.W_b, z=z, workspace=ws,
                                                       stream=stream), bw["broadcast"], "hbm"),
            "transition": (lambda: nt.nt_pair_transition(part, z, wd.ln_gamma, wd.ln_beta, wd.W1, wd.b1, wd.W2,
                                                         wd.b2, out=zt, stream=stream), bw["transition"], "tensor"),
            "reduce": (lambda: nt.nt_pair_reduce(part, zt, wd.W_g, wd.b_g, s_in=s, m=m, s_out=so, stream=stream),
                       bw["reduce"], "hbm"),
            "block": (lambda: nt.block_forward(part, s, wd, z=z, workspace=ws, s_out=so, stream=stream),
                      {k: sum(v[k] for v in bw.values()) for k in ("bytes", "flops")}, "tensor"),
            # one pass: z~ written once (256 B/cell), singles-sized traffic besides
            "fused": (lambda: nt.nt_pair_block_fused(part, s, s, wd, z=zt, m=m, s_out=so, workspace=wsf,
                                                     stream=stream),
                      {"bytes": part.P * cfg.C_z * es + bw["reduce"]["bytes"] - part.P * cfg.C_z * es,
                       "flops": bw["transition"]["flops"]}, "tensor"),
        }
        # the Eq. 5 loss and the block's backward (CUDA cores): the forward's
        # outputs are made once, outside the timed calls
        zb, mb, sob = nt.block_forward(part, s, wd)
        bound_b = "tensor" if backward_route(cfg) == "tensor" else "fma"
        # per cell: A recomputed, dH, dY, dW1, dW2 (five C_z x H_t products)
        work_b = {"bytes": 0, "flops": 5 * 2 * cfg.C_z * cfg.H_t * part.P}
        if args.only == "backward":
            lws = torch.empty(nt.nt_pair_block_loss_backward_workspace_bytes(nt._dtype(s), part.T, part.P, cfg.C_s,
                                                                             cfg.C_z, cfg.H_t),
                              dtype=torch.uint8, device=dev)
            lossb = torch.empty(1, dtype=torch.float32, device=dev)
            fns["backward"] = (lambda: nt.nt_pair_block_loss_backward(part, s, wd, mb, sob, zb, loss=lossb,
                                                                      workspace=lws, stream=stream),
                               work_b, bound_b)
        if args.only == "backward_two_calls":
            bws = torch.empty(nt.nt_pair_block_backward_workspace_bytes(nt._dtype(s), part.T, part.P, cfg.C_z,
                                                                        cfg.H_t),
                              dtype=torch.uint8, device=dev)

            def backward_step():
                _, ds_out, dz = nt.nt_pair_block_loss(part, sob, zb, stream=stream)
                nt.nt_pair_block_backward(part, s, wd, mb, ds_out, dz, workspace=bws, stream=stream)
            fns["backward_two_calls"] = (backward_step, work_b, bound_b)
        if args.swiglu:
            sw = wl.make_swiglu_weights(cfg.C_z, cfg.H_t, cfg.dtype)
            d = lambda t: None if t is None else t.to(dev)
            g1, be1, W1s, W3s, W2s = d(sw.ln_gamma), d(sw.ln_beta), d(sw.W1), d(sw.W3), d(sw.W2)
            # gate and value GEMMs (2 x 2 C_z H_t) plus the output GEMM (2 H_t C_z) per cell
            fns["transition"] = (lambda: nt.nt_pair_transition_swiglu(part, z, g1, be1, W1s, None, W3s, None, W2s,
                                                                       None, out=zt, stream=stream),
                                 {"bytes": bw["transition"]["bytes"] + cfg.H_t * cfg.C_z * es,
                                  "flops": 6 * cfg.C_z * cfg.H_t * part.P}, "tensor")
        fn, w, bound = fns[args.only]
        name = cfg.name + ("_swiglu" if args.swiglu and args.only == "transition" else "")
    for _ in range(args.warmup):
        flush.fill_(0.0)
        fn()
    torch.cuda.synchronize()
    times = []
    for i in range(args.steps):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    nt.nt_device_status(stream)
    ms = float(np.mean([a.elapsed_time(b) for a, b in times]))
    out = {"kernel": args.only, "workload": name, "ms": ms, "steps": args.steps}
    if bound == "tensor":
        out.update({"bound": "tensor", "achieved": w["flops"] / ms / 1e9, "unit": "TFLOP/s",
                    "peak": peaks["bf16_tflops"]})
    elif bound == "hbm":
        out.update({"bound": "hbm", "achieved": w["bytes"] / ms / 1e6, "unit": "GB/s", "peak": peaks["hbm_gbs"]})
    elif bound == "fma":
        fp32_peak = fp32_fma_tflops(dev, peaks)
        out.update({"bound": "alu", "achieved": w["flops"] / ms / 1e9, "unit": "TFLOP/s", "peak": fp32_peak,
                    "peak_source": "fp32 FMA: 128 per SM per clock x 2 flop x SMs x max SM clock"})
    if "peak" in out:
        out["frac"] = out["achieved"] / out["peak"]
        out.setdefault("peak_source", peak_src)
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    choices=["partition", "broadcast", "transition", "reduce", "block", "fused", "attention",
                             "backward", "backward_two_calls", "packing", "padsweep", "rect"],
                    help="time one call on one workload instead of the whole step; 'packing' and "
                         "'padsweep' print the packed-vs-padded reports")
    ap.add_argument("--workload", default="pairformer", choices=sorted(WORKLOADS))
    ap.add_argument("--causal", action="store_true", help="with --only attention: the causal mask")
    ap.add_argument("--swiglu", action="store_true", help="with --only transition: the SwiGLU update")
    ap.add_argument("--backward", action="store_true", help="with --only attention: the backward (dq, dk, dv)")
    args = ap.parse_args()
    if args.only == "packing":
        nt, dev, stream, flush = _report_setup()
        for line in run_packing(nt, dev, stream, flush, args.steps):
            print(json.dumps(dict(report="packing", **line)), flush=True)
        return
    if args.only == "padsweep":
        nt, dev, stream, flush = _report_setup()
        for line in run_padsweep(nt, dev, stream, flush, args.steps, load_peaks()[0]):
            print(json.dumps(dict(report="padsweep", **line)), flush=True)
        return
    if args.only == "rect":
        run_rect(args)
        return
    if args.only:
        run_only(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_gpu(args, rank, world, local_rank)
    if line is not None:
        if not args.no_cpu_baseline:
            v, smp = oracle_block_sample()
            av, asmp = oracle_attn_sample()
            line["cpu_baseline"] = {"value": v, "unit": "pair cells/s", "cores": cpu_cores(),
                                    "threads": cpu_threads(), "kind": "oracle", "sample": smp,
                                    "attn_tflops": av, "attn_sample": asmp}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
