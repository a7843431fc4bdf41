"""The multi-rank path on CPU with gloo, world size 2: sample sharding with
no exchange reproduces the single-process oracle, and the benchmark's
max-over-ranks reduction and whole-job throughput behave as stated."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from variable_length_batching_gb300.sharding import shard_rows, shard_samples


def test_shard_samples_balanced_and_complete():
    lengths = [1024, 768, 512, 384, 256, 192, 128, 64]
    for world in (1, 2, 3, 4, 8):
        shards = shard_samples(lengths, world)
        assert sorted(i for s in shards for i in s) == list(range(len(lengths)))
        loads = [sum(lengths[i] ** 2 for i in s) for s in shards]
        # LPT bound: max load <= mean + largest single item
        assert max(loads) <= sum(loads) / world + max(l ** 2 for l in lengths)
    assert shard_samples([5, 0, 3], 2) == [[0], [1, 2]]
    assert shard_rows([2, 3, 1], [2, 0]) == [5, 0, 1]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from oracle import block as oblock
        from _helpers import oracle_weights, f64
        from variable_length_batching_gb300 import workloads as wl
        # timings: the max over ranks, whatever each rank measured
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 2.0], world)
        assert got == [float(world), 5.0, 2.0]
        thr = bench.job_throughput(100, world, got[0])
        assert abs(thr - world * 100 / (world * 1e-3)) < 1e-6
        # sample sharding: each rank runs the oracle block on its own samples only
        cfg = wl.TINY_FP32
        inp = wl.make_block_inputs(cfg, lengths=[9, 3, 7, 1, 12, 5], biases=True)
        w = oracle_weights(inp.blocks[0])
        s = f64(inp.s)
        mine = shard_samples(inp.lengths, world)[rank]
        rows = shard_rows(inp.lengths, mine)
        res = oblock.block_packed([int(inp.lengths[i]) for i in mine], s[rows], w)
        gathered = [None] * world
        dist.all_gather_object(gathered, (rows, res.s_out))
        if rank == 0:
            full = oblock.block_packed(inp.lengths, s, w)
            merged = np.zeros_like(full.s_out)
            for r_rows, r_out in gathered:
                merged[r_rows] = r_out
            out.put(float(np.abs(merged - full.s_out).max()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert q.get(timeout=10) == 0.0
