"""The C-ABI library loads here (no GPU) and exports every symbol the header
declares; host-side argument checks reject bad calls before any CUDA call."""
import ctypes
import os
import re

import pytest

from variable_length_batching_gb300 import build as nt_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nt.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nt_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    path = nt_build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("nt_partition_build", "nt_partition_rows", "nt_pair_broadcast", "nt_pair_transition",
              "nt_pair_reduce", "nt_varlen_attn", "nt_varlen_attn_qk", "nt_device_status", "nt_status_str",
              "nt_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), n


def test_binding_covers_every_declaration():
    from variable_length_batching_gb300 import nt
    assert set(nt.SIGNATURES) == set(declared_functions())


def test_status_strings(L):
    L.nt_status_str.restype = ctypes.c_char_p
    assert L.nt_status_str(0) == b"NT_OK"
    assert L.nt_status_str(1) == b"NT_ERR_INVALID"
    assert L.nt_status_str(5) == b"NT_ERR_TIMEOUT"
    assert L.nt_status_str(99) == b"NT_ERR_UNKNOWN"


def test_workspace_bytes(L):
    L.nt_pair_broadcast_workspace_bytes.restype = ctypes.c_size_t
    L.nt_pair_broadcast_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32]
    assert L.nt_pair_broadcast_workspace_bytes(1031, 128) == 2 * 1031 * 128 * 4
    assert L.nt_pair_broadcast_workspace_bytes(-1, 128) == 0


def test_block_backward_workspace_bytes():
    """The CUDA-core route needs (5 T + P) C_z fp32 words (rounded up to 256
    bytes); the bf16 tensor-core route (C_z = 128, H_t % 128 == 0) adds its
    cell rows: [hi | lo] LN(z) and dP~ ([P, C_z] bf16-sized), H and dA
    ([P, H_t] bf16 each) and the per-cell statistics, so at least that."""
    from variable_length_batching_gb300 import nt
    T, P, C, H = 1031, 157023, 128, 512
    base = -(-(5 * T + P) * C * 4 // 256) * 256
    assert nt.nt_pair_block_backward_workspace_bytes(nt.NT_F32, T, P, C, H) == base
    assert nt.nt_pair_block_backward_workspace_bytes(nt.NT_BF16, T, P, 64, 256) == -(-(5 * T + P) * 64 * 4 // 256) * 256
    tc = nt.nt_pair_block_backward_workspace_bytes(nt.NT_BF16, T, P, C, H)
    assert tc >= base + P * (2 * C * 2 + C * 2 + 2 * H * 2 + 8)
    assert nt.nt_pair_block_backward_workspace_bytes(nt.NT_BF16, -1, P, C, H) == 0


def test_block_loss_backward_workspace_bytes():
    """The fused loss + backward needs the loss's partial sums, dL/dX~ ([T,
    C_s] fp32) and the backward's workspace; dL/dz~ ([P, C_z] fp32) as well,
    except on the tensor-core route, which forms it from z~."""
    from variable_length_batching_gb300 import nt
    T, P, Cs, C, H = 1031, 157023, 384, 128, 512
    loss_ws = int(nt.lib().nt_pair_block_loss_workspace_bytes())
    for dt, Cz, Ht, dz in ((nt.NT_BF16, C, H, 0), (nt.NT_F32, C, H, P * C * 4), (nt.NT_BF16, 64, 256, P * 64 * 4)):
        got = nt.nt_pair_block_loss_backward_workspace_bytes(dt, T, P, Cs, Cz, Ht)
        bwd = nt.nt_pair_block_backward_workspace_bytes(dt, T, P, Cz, Ht)
        assert bwd + loss_ws + T * Cs * 4 + dz <= got <= bwd + loss_ws + T * Cs * 4 + dz + 3 * 256
    assert nt.nt_pair_block_loss_backward_workspace_bytes(nt.NT_BF16, T, P, -1, C, H) == 0


def test_host_side_rejections(L):
    """Calls that must fail on argument checks alone (nothing reaches CUDA)."""
    from variable_length_batching_gb300 import nt
    lib = nt.lib()
    part = nt.nt_partition()
    P = ctypes.byref(part)
    fake = ctypes.c_void_p(0x1000)       # never dereferenced: the checks fire first
    odd = ctypes.c_void_p(0x1008)
    # NULL output struct / negative B
    assert lib.nt_partition_build(fake, 4, fake, fake, fake, None, None) == 1
    assert lib.nt_partition_build(fake, -1, fake, fake, fake, P, None) == 1
    # NULL partition
    assert lib.nt_pair_transition(None, 1, fake, fake, 128, 512, fake, fake, 1e-5, fake, None,
                                  fake, None, None) == 1
    # partition without row splits
    part.B, part.T, part.P, part.max_len = 2, 5, 13, 3
    part.lengths = part.cu_seqlens = part.pair_off = 0x1000
    assert lib.nt_pair_broadcast(P, 1, fake, fake, 384, fake, fake, 128, fake, fake, 1 << 20, None) == 1
    part.row_start = part.row_sample = 0x1000
    # inconsistent totals: P > T * max_len
    part.P = 100
    assert lib.nt_pair_reduce(P, 1, fake, 128, fake, None, None, None, None, 0, None) == 1
    part.P = 13
    # the reduce fused with the loss: W_g and the loss are required, and its workspace
    rl = lib.nt_pair_reduce_loss
    ws = int(lib.nt_pair_reduce_loss_workspace_bytes())
    assert ws >= 8 * (2 * 1024 + 8192)
    assert rl(P, 1, fake, 128, fake, None, None, fake, fake, 384, fake, fake, ws, None) == 1
    assert rl(P, 1, fake, 128, fake, fake, None, fake, fake, 384, None, fake, ws, None) == 1
    assert rl(P, 1, fake, 128, fake, fake, None, fake, fake, 384, fake, fake, 16, None) == 1
    # width not a multiple of 8 in bf16 -> unsupported
    assert lib.nt_pair_broadcast(P, 1, fake, fake, 384, fake, fake, 12, fake, fake, 1 << 20, None) == 2
    # misaligned pointer
    assert lib.nt_pair_broadcast(P, 1, odd, fake, 384, fake, fake, 128, fake, fake, 1 << 20, None) == 1
    # workspace too small
    assert lib.nt_pair_broadcast(P, 1, fake, fake, 384, fake, fake, 128, fake, fake, 16, None) == 1
    # bad dtype
    assert lib.nt_pair_transition(P, 7, fake, fake, 128, 512, fake, fake, 1e-5, fake, None, fake,
                                  None, None) == 1
    # attention backward: bad head width, bad causal flag
    bw = lib.nt_varlen_attn_bwd
    assert bw(1, fake, fake, fake, fake, fake, fake, fake, fake, 1, 64, 64, 64, 64, 1, 48, 0.125, 0, fake, fake,
              fake, fake, 1 << 20, None) == 2
    assert bw(1, fake, fake, fake, fake, fake, fake, fake, fake, 1, 64, 64, 64, 64, 1, 64, 0.125, 3, fake, fake,
              fake, fake, 1 << 20, None) == 1
    # a negative max length
    assert bw(1, fake, fake, fake, fake, fake, fake, fake, fake, 1, 64, 64, 64, -1, 1, 64, 0.125, 0, fake, fake,
              fake, fake, 1 << 20, None) == 1
    # more cells than 32-bit copy coordinates reach
    assert lib.nt_pair_transition_cells(2**31, 1, fake, fake, 128, 512, fake, fake, 1e-5, fake, None, None, None,
                                        fake, None, None) == 3
    # the wait self-test: bad mode, a limit of 0 or above 2 s, a delay above 2 s, NULL or misaligned result
    sw = lib.nt_selftest_bounded_wait
    assert sw(3, 0, 10**6, fake, None) == 1
    assert sw(1, 0, 0, fake, None) == 1
    assert sw(1, 0, 2 * 10**9 + 1, fake, None) == 1
    assert sw(0, 2 * 10**9 + 1, 10**6, fake, None) == 1
    assert sw(1, 0, 10**6, None, None) == 1
    assert sw(1, 0, 10**6, ctypes.c_void_p(0x1004), None) == 1
    # SwiGLU without its value projection
    assert lib.nt_pair_transition_swiglu(P, 1, fake, fake, 128, 512, fake, fake, 1e-5, fake, None, None, None,
                                         fake, None, None) == 1
    # partition with row splits in one call: NULL out, negative B or capacity, NULL row buffers
    pw = lib.nt_partition_build_with_rows
    assert pw(fake, 4, 16, fake, fake, fake, fake, fake, None, None) == 1
    assert pw(fake, -1, 16, fake, fake, fake, fake, fake, P, None) == 1
    assert pw(fake, 4, -1, fake, fake, fake, fake, fake, P, None) == 1
    assert pw(fake, 4, 16, fake, fake, fake, None, fake, P, None) == 1
    # transition over a cell range: negative count, bad dtype, misaligned slice; zero cells is a no-op
    tc = lib.nt_pair_transition_cells
    assert tc(-1, 1, fake, fake, 128, 512, fake, fake, 1e-5, fake, None, None, None, fake, None, None) == 1
    assert tc(10, 7, fake, fake, 128, 512, fake, fake, 1e-5, fake, None, None, None, fake, None, None) == 1
    assert tc(10, 1, odd, fake, 128, 512, fake, fake, 1e-5, fake, None, None, None, fake, None, None) == 1
    assert tc(0, 1, fake, fake, 128, 512, fake, fake, 1e-5, fake, None, None, None, fake, None, None) == 0
    # W_g without s_out
    assert lib.nt_pair_reduce(P, 1, fake, 128, fake, fake, None, None, None, 384, None) == 1
    # attention: T > 0 without segments; bad head count; T beyond int32
    assert lib.nt_varlen_attn(1, fake, fake, fake, fake, 0, 64, 64, 12, 64, 0.125, fake, None, None, 0, None) == 1
    assert lib.nt_varlen_attn(1, fake, fake, fake, fake, 1, 64, 64, 0, 64, 0.125, fake, None, None, 0, None) == 1
    assert lib.nt_varlen_attn(1, fake, fake, fake, fake, 1, 1 << 31, 64, 1, 64, 0.125, fake, None, None, 0, None) == 3
    # an empty stream is a no-op success
    assert lib.nt_varlen_attn(1, None, None, None, None, 0, 0, 0, 12, 64, 0.125, None, None, None, 0, None) == 0
    # scale must be finite and > 0
    for bad in (0.0, -0.125, float("inf"), float("nan")):
        assert lib.nt_varlen_attn(1, fake, fake, fake, fake, 1, 64, 64, 1, 64, bad, fake, None, None, 0, None) == 1
    # qk form: causal flag 0/1 only; T_k beyond int32; key pointers needed when T_k > 0
    qk = lib.nt_varlen_attn_qk
    assert qk(1, fake, fake, fake, fake, fake, 1, 64, 64, 64, 1, 64, 0.125, 2, fake, None, None, 0, None) == 1
    assert qk(1, fake, fake, fake, fake, fake, 1, 64, 1 << 31, 64, 1, 64, 0.125, 0, fake, None, None, 0, None) == 3
    assert qk(1, fake, None, None, fake, fake, 1, 64, 32, 64, 1, 64, 0.125, 0, fake, None, None, 0, None) == 1
    assert qk(1, fake, fake, fake, fake, fake, 1, -1, 32, 64, 1, 64, 0.125, 0, fake, None, None, 0, None) == 1
    assert qk(1, None, None, None, None, None, 0, 0, 0, 0, 4, 64, 0.125, 1, None, None, None, 0, None) == 0
    # a workspace smaller than the stated size, or misaligned
    assert lib.nt_varlen_attn(1, fake, fake, fake, fake, 1, 64, 64, 1, 64, 0.125, fake, None, fake, 4, None) == 1
    assert lib.nt_varlen_attn(1, fake, fake, fake, fake, 1, 64, 64, 1, 64, 0.125, fake, None, odd, 256, None) == 1
    assert lib.nt_varlen_attn_workspace_bytes() >= 4
    assert lib.nt_last_error()  # a detail string was recorded
