"""GPU parity of nt_pair_reduce_loss: the column mean and g projection of
"DanLing NestedTensor" Eq. 1 (third line) with the Eq. 5 loss of Appendix
A.1 in one call that reads z~ once.  m and s_out equal nt_pair_reduce's bit
for bit; the loss equals nt_pair_block_loss's up to the order of its sums
and the oracle's Eq. 5 within the loss's usual bound."""
import numpy as np
import pytest
import torch

from _helpers import f64, to_np
from oracle import block_backward as obwd

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def nt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from variable_length_batching_gb300 import build, nt as ntmod
    build.build()
    return ntmod


@pytest.mark.parametrize("dtype,C_s,C_z,lengths", [
    (torch.bfloat16, 384, 128, [37, 1, 0, 70, 256, 5]),     # the reduce's squares fused
    (torch.float32, 32, 16, [5, 0, 9, 1, 33]),              # fp32, fused
    (torch.float32, 24, 12, [5, 0, 9, 1, 33]),              # fp32, C_z not a multiple of 8: z~ read again
])
def test_reduce_loss_matches_two_calls_and_oracle(nt, dtype, C_s, C_z, lengths):
    g = torch.Generator().manual_seed(11)
    T, P = sum(lengths), sum(n * n for n in lengths)
    z = torch.randn(P, C_z, generator=g).to(dtype).to(DEV)
    s_in = torch.randn(T, C_s, generator=g).to(dtype).to(DEV)
    W_g = (torch.randn(C_s, C_z, generator=g) / C_z ** 0.5).to(dtype).to(DEV)
    b_g = torch.randn(C_s, generator=g).to(DEV)
    part = nt.nt_partition_build(torch.tensor(lengths, dtype=torch.int32, device=DEV))
    m1, s1 = nt.nt_pair_reduce(part, z, W_g, b_g, s_in=s_in)
    l1, _, _ = nt.nt_pair_block_loss(part, s1, z, want_grads=False)
    m2, s2, l2 = nt.nt_pair_reduce_loss(part, z, W_g, b_g, s_in=s_in)
    m3, s3, l3 = nt.nt_pair_reduce_loss(part, z, W_g, b_g, s_in=s_in)
    torch.cuda.synchronize()
    nt.nt_device_status()
    assert torch.equal(m1, m2) and torch.equal(s1, s2)
    assert torch.equal(l2, l3)                                  # fixed order: reproducible
    a, b = float(l1.item()), float(l2.item())
    assert abs(a - b) <= 1e-6 * abs(a), (a, b)
    ref = obwd.eq5_loss(lengths, f64(s2.cpu()), f64(z.cpu()))
    assert abs(b - ref) <= 1e-5 * abs(ref), (b, ref)


def test_reduce_loss_empty_batch(nt):
    part = nt.nt_partition_build(torch.zeros(3, dtype=torch.int32, device=DEV))
    z = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    s_in = torch.empty(0, 384, dtype=torch.bfloat16, device=DEV)
    W_g = torch.zeros(384, 128, dtype=torch.bfloat16, device=DEV)
    m = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    s_out = torch.empty(0, 384, dtype=torch.bfloat16, device=DEV)
    _, _, loss = nt.nt_pair_reduce_loss(part, z, W_g, None, s_in=s_in, m=m, s_out=s_out)
    torch.cuda.synchronize()
    assert float(loss.item()) == 0.0
