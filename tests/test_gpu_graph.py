"""GPU parity of BlockGraph, the host-to-host block step replayed from a
CUDA graph ("DanLing NestedTensor" Eq. 1): its z~ and s_out equal the eager
three calls' bit for bit (the transition runs in slices of cells, which is
cell-for-cell identical), on the first step (eager pass plus capture), on
replays, and after new lengths force a new capture."""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

from variable_length_batching_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def mods():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_batching_gb300 import build, graph, nt as ntmod
    build.build()
    return ntmod, graph


def _eager(nt, inp, wd):
    part = nt.nt_partition_build(torch.as_tensor(np.asarray(inp.lengths, dtype=np.int32)).to(DEV))
    z, m, s_out = nt.block_forward(part, inp.s.to(DEV), wd)
    return z.cpu(), s_out.cpu()


@pytest.mark.parametrize("slices,growth", [(3, 2.0), (4, 1.0), (1, 1.0)])
def test_block_graph_matches_eager(mods, slices, growth):
    nt, graph = mods
    cfg = wl.PAIRFORMER_BF16
    inp = wl.make_block_inputs(cfg, biases=True)
    w = inp.blocks[0]
    g = lambda t: None if t is None else t.to(DEV).contiguous()
    wd = SimpleNamespace(W_a=g(w.W_a), W_b=g(w.W_b), ln_gamma=g(w.ln_gamma), ln_beta=g(w.ln_beta), W1=g(w.W1),
                         b1=g(w.b1), W2=g(w.W2), b2=g(w.b2), W_g=g(w.W_g), b_g=g(w.b_g))
    runner = graph.BlockGraph(wd, slices=slices, growth=growth)
    lengths = torch.as_tensor(np.asarray(inp.lengths, dtype=np.int32)).pin_memory()
    s = inp.s.pin_memory()
    z_ref, s_ref = _eager(nt, inp, wd)
    for _ in range(3):                                   # capture, then two replays
        z_h, s_h = runner.run(lengths, s)
        assert torch.equal(z_h, z_ref) and torch.equal(s_h, s_ref)
    # other lengths: a new capture
    inp2 = wl.make_block_inputs(cfg, lengths=[64, 1, 200, 0, 37, 5, 128, 90], biases=True)
    z2_ref, s2_ref = _eager(nt, inp2, wd)
    for _ in range(2):
        z_h, s_h = runner.run(torch.as_tensor(np.asarray(inp2.lengths, dtype=np.int32)).pin_memory(),
                              inp2.s.pin_memory())
        assert torch.equal(z_h, z2_ref) and torch.equal(s_h, s2_ref)
    nt.nt_device_status()


def test_block_graph_pipelined_steps(mods):
    """Steps in flight two at a time (submit the next before waiting for the
    previous): each step's z~ and s_out equal its own eager block's, bit for
    bit, though its compute overlaps the previous step's read-back."""
    nt, graph = mods
    cfg = wl.PAIRFORMER_BF16
    base = wl.make_block_inputs(cfg, biases=True)
    # the same lengths (one key: the graphs are reused), other singles
    inps = [base] + [wl.make_block_inputs(cfg, lengths=base.lengths, biases=True, seed=sd) for sd in (1, 2, 3)]
    w = inps[0].blocks[0]
    g = lambda t: None if t is None else t.to(DEV).contiguous()
    wd = SimpleNamespace(W_a=g(w.W_a), W_b=g(w.W_b), ln_gamma=g(w.ln_gamma), ln_beta=g(w.ln_beta), W1=g(w.W1),
                         b1=g(w.b1), W2=g(w.W2), b2=g(w.b2), W_g=g(w.W_g), b_g=g(w.b_g))
    refs = []
    for x in inps:
        x.blocks = inps[0].blocks           # the same weights, other singles
        refs.append(_eager(nt, x, wd))
    runner = graph.BlockGraph(wd, depth=2)
    lengths = torch.as_tensor(np.asarray(inps[0].lengths, dtype=np.int32)).pin_memory()
    hs = [x.s.pin_memory() for x in inps]
    tickets, got = [], []
    for i, s in enumerate(hs + hs):          # eight steps, two passes over the four inputs
        tickets.append(runner.submit(lengths, s))
        if i >= 1:
            z_h, s_h = runner.wait(tickets[i - 1])
            got.append((z_h.clone(), s_h.clone()))
    z_h, s_h = runner.wait(tickets[-1])
    got.append((z_h.clone(), s_h.clone()))
    for i, (z_h, s_h) in enumerate(got):
        z_ref, s_ref = refs[i % 4]
        assert torch.equal(z_h, z_ref) and torch.equal(s_h, s_ref), f"step {i}"
    with pytest.raises(ValueError):
        runner.wait(tickets[0])              # reused two submissions later
    nt.nt_device_status()


def test_block_graph_loss_readback(mods):
    """readback="loss": each step reads back the Eq. 5 loss of its two
    outputs ("DanLing NestedTensor" Appendix A.1), computed on the device in
    the captured graph (the reduce fused with the loss), and s_out; both
    equal the same calls made eagerly bit for bit, over pipelined steps with
    other singles and after new lengths, and the loss equals the two-pass
    nt_pair_block_loss up to the order of its sums."""
    nt, graph = mods
    cfg = wl.PAIRFORMER_BF16
    base = wl.make_block_inputs(cfg, biases=True)
    inps = [base] + [wl.make_block_inputs(cfg, lengths=base.lengths, biases=True, seed=sd) for sd in (1, 2)]
    w = base.blocks[0]
    g = lambda t: None if t is None else t.to(DEV).contiguous()
    wd = SimpleNamespace(W_a=g(w.W_a), W_b=g(w.W_b), ln_gamma=g(w.ln_gamma), ln_beta=g(w.ln_beta), W1=g(w.W1),
                         b1=g(w.b1), W2=g(w.W2), b2=g(w.b2), W_g=g(w.W_g), b_g=g(w.b_g))

    def eager_loss(x):
        # the graph's calls, eagerly: broadcast, transition, then the reduce
        # fused with the loss; and the two-pass loss up to summation order
        part = nt.nt_partition_build(torch.as_tensor(np.asarray(x.lengths, dtype=np.int32)).to(DEV))
        s = x.s.to(DEV)
        z = nt.nt_pair_broadcast(part, s, s, wd.W_a, wd.W_b)
        nt.nt_pair_transition(part, z, wd.ln_gamma, wd.ln_beta, wd.W1, wd.b1, wd.W2, wd.b2, out=z)
        _, s_out, loss = nt.nt_pair_reduce_loss(part, z, wd.W_g, wd.b_g, s_in=s)
        two_pass, _, _ = nt.nt_pair_block_loss(part, s_out, z, want_grads=False)
        assert abs(float(loss.item()) - float(two_pass.item())) <= 1e-6 * abs(float(two_pass.item()))
        return loss.cpu(), s_out.cpu()

    refs = [eager_loss(x) for x in inps]
    runner = graph.BlockGraph(wd, depth=2, readback="loss")
    assert runner.slices == 1
    lengths = torch.as_tensor(np.asarray(base.lengths, dtype=np.int32)).pin_memory()
    hs = [x.s.pin_memory() for x in inps]
    tickets, got = [], []
    for i, s in enumerate(hs + hs):
        tickets.append(runner.submit(lengths, s))
        if i >= 1:
            l_h, s_h = runner.wait(tickets[i - 1])
            got.append((l_h.clone(), s_h.clone()))
    l_h, s_h = runner.wait(tickets[-1])
    got.append((l_h.clone(), s_h.clone()))
    for i, (l_h, s_h) in enumerate(got):
        l_ref, s_ref = refs[i % 3]
        assert torch.equal(l_h, l_ref) and torch.equal(s_h, s_ref), f"step {i}"
    inp2 = wl.make_block_inputs(cfg, lengths=[64, 1, 200, 0, 37, 5, 128, 90], biases=True)
    inp2.blocks = base.blocks
    l2_ref, s2_ref = eager_loss(inp2)
    l_h, s_h = runner.run(torch.as_tensor(np.asarray(inp2.lengths, dtype=np.int32)).pin_memory(), inp2.s.pin_memory())
    assert torch.equal(l_h, l2_ref) and torch.equal(s_h, s2_ref)
    with pytest.raises(ValueError):
        graph.BlockGraph(wd, readback="z")
    nt.nt_device_status()


def test_block_graph_shapes_change_in_flight(mods):
    """Pipelined steps whose (B, T, P) change from one submission to the next
    and back (each change drains the pipeline and captures anew; the input
    slots are reallocated when B or T changes, kept when only the values
    do): every step's z~ and s_out equal the eager calls' bit for bit."""
    nt, graph = mods
    cfg = wl.PAIRFORMER_BF16
    base = wl.make_block_inputs(cfg, lengths=[37, 1, 0, 70], biases=True)
    w = base.blocks[0]
    g = lambda t: None if t is None else t.to(DEV).contiguous()
    wd = SimpleNamespace(W_a=g(w.W_a), W_b=g(w.W_b), ln_gamma=g(w.ln_gamma), ln_beta=g(w.ln_beta), W1=g(w.W1),
                         b1=g(w.b1), W2=g(w.W2), b2=g(w.b2), W_g=g(w.W_g), b_g=g(w.b_g))
    shapes = [[37, 1, 0, 70], [37, 1, 0, 70], [5, 90, 33], [37, 1, 0, 70], [70, 1, 0, 37], [5, 90, 33], [5, 90, 33]]
    inps = []
    for i, lengths in enumerate(shapes):
        x = wl.make_block_inputs(cfg, lengths=lengths, biases=True, seed=20 + i)
        x.blocks = base.blocks
        inps.append(x)
    refs = [_eager(nt, x, wd) for x in inps]
    runner = graph.BlockGraph(wd, slices=2, growth=2.0, depth=2)
    tickets, got = [], []
    for i, x in enumerate(inps):
        tickets.append(runner.submit(torch.as_tensor(np.asarray(x.lengths, dtype=np.int32)).pin_memory(),
                                     x.s.pin_memory()))
        if i >= 1:
            z_h, s_h = runner.wait(tickets[i - 1])
            got.append((z_h.clone(), s_h.clone()))
    z_h, s_h = runner.wait(tickets[-1])
    got.append((z_h.clone(), s_h.clone()))
    for i, ((z_h, s_h), (z_ref, s_ref)) in enumerate(zip(got, refs)):
        assert torch.equal(z_h, z_ref) and torch.equal(s_h, s_ref), f"step {i} ({shapes[i]})"
    nt.nt_device_status()
