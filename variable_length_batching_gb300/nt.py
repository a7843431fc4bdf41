"""Thin Python binding of libnt (``include/nt.h``).

Argument marshalling only: torch tensors supply device memory and the
current CUDA stream; every step of the block and of varlen attention runs in
the library's kernels.  Functions keep the C names.  If ``libnt.so`` is
missing or a call fails, an exception is raised -- there is no other path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnt.so")

NT_F32, NT_BF16 = 0, 1
STATUS = {0: "NT_OK", 1: "NT_ERR_INVALID", 2: "NT_ERR_UNSUPPORTED", 3: "NT_ERR_OVERFLOW",
          4: "NT_ERR_CUDA", 5: "NT_ERR_TIMEOUT", 6: "NT_ERR_DEVICE_CHECK"}


class NTError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {detail}")
        self.status = status


class nt_partition(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int64), ("P", ctypes.c_int64),
                ("max_len", ctypes.c_int32), ("lengths", ctypes.c_void_p),
                ("cu_seqlens", ctypes.c_void_p), ("pair_off", ctypes.c_void_p),
                ("row_start", ctypes.c_void_p), ("row_sample", ctypes.c_void_p),
                ("col_lengths", ctypes.c_void_p), ("col_cu_seqlens", ctypes.c_void_p),
                ("T_cols", ctypes.c_int64), ("max_col_len", ctypes.c_int32)]


_lib = None

_P, _I32, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_PP = ctypes.POINTER(nt_partition)
SIGNATURES = {
    "nt_partition_build": (_I32, [_P, _I32, _P, _P, _P, _PP, _P]),
    "nt_partition_build_rect": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _PP, _P]),
    "nt_partition_rows": (_I32, [_PP, _P, _P, _P]),
    "nt_pair_broadcast_workspace_bytes": (_SZ, [_I64, _I32]),
    "nt_pair_broadcast_workspace_bytes_rect": (_SZ, [_I64, _I64, _I32]),
    "nt_pair_broadcast": (_I32, [_PP, _I32, _P, _P, _I32, _P, _P, _I32, _P, _P, _SZ, _P]),
    "nt_pair_broadcast_noalloc": (_I32, [_PP, _I32, _P, _P, _I32, _P, _P, _I32, _P, _P]),
    "nt_pair_transition": (_I32, [_PP, _I32, _P, _P, _I32, _I32, _P, _P, _F, _P, _P, _P, _P, _P]),
    "nt_pair_transition_swiglu": (_I32, [_PP, _I32, _P, _P, _I32, _I32, _P, _P, _F, _P, _P, _P, _P, _P, _P,
                                         _P]),
    "nt_partition_build_with_rows": (_I32, [_P, _I32, _I64, _P, _P, _P, _P, _P, _PP, _P]),
    "nt_pair_transition_cells": (_I32, [_I64, _I32, _P, _P, _I32, _I32, _P, _P, _F, _P, _P, _P, _P, _P, _P,
                                        _P]),
    "nt_pair_reduce": (_I32, [_PP, _I32, _P, _I32, _P, _P, _P, _P, _P, _I32, _P]),
    "nt_pair_block_fused_workspace_bytes": (_SZ, [_I64, _I64, _I32]),
    "nt_pair_block_fused": (_I32, [_PP, _I32, _P, _P, _I32, _P, _P, _I32, _I32, _P, _P, _F, _P, _P, _P, _P, _P, _P,
                                   _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "nt_pair_reduce_loss_workspace_bytes": (_SZ, []),
    "nt_pair_reduce_loss": (_I32, [_PP, _I32, _P, _I32, _P, _P, _P, _P, _P, _I32, _P, _P, _SZ, _P]),
    "nt_pair_block_loss_workspace_bytes": (_SZ, []),
    "nt_pair_block_loss": (_I32, [_PP, _I32, _P, _I32, _P, _I32, _P, _P, _P, _P, _SZ, _P]),
    "nt_pair_block_backward_workspace_bytes": (_SZ, [_I32, _I64, _I64, _I32, _I32]),
    "nt_pair_block_backward": (_I32, [_PP, _I32, _P, _I32, _P, _P, _I32, _I32, _P, _P, _F, _P, _P, _P, _P, _P, _P,
                                      _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "nt_pair_block_loss_backward_workspace_bytes": (_SZ, [_I32, _I64, _I64, _I32, _I32, _I32]),
    "nt_pair_block_loss_backward": (_I32, [_PP, _I32, _P, _I32, _P, _P, _I32, _I32, _P, _P, _F, _P, _P, _P, _P,
                                           _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                           _P]),
    "nt_varlen_attn_workspace_bytes": (_SZ, []),
    "nt_varlen_attn": (_I32, [_I32, _P, _P, _P, _P, _I32, _I64, _I32, _I32, _I32, _F, _P, _P, _P, _SZ, _P]),
    "nt_varlen_attn_qk": (_I32, [_I32, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I32, _I32, _I32, _F, _I32,
                                 _P, _P, _P, _SZ, _P]),
    "nt_varlen_attn_bwd_workspace_bytes": (_SZ, [_I64, _I32]),
    "nt_varlen_attn_bwd": (_I32, [_I32, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I32, _I32, _I32, _I32,
                                  _F, _I32, _P, _P, _P, _P, _SZ, _P]),
    "nt_device_status": (_I32, [_P]),
    "nt_selftest_bounded_wait": (_I32, [_I32, ctypes.c_uint64, ctypes.c_uint64, _P, _P]),
    "nt_status_str": (ctypes.c_char_p, [_I32]),
    "nt_last_error": (ctypes.c_char_p, []),
}


def lib():
    """Load libnt.so once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m variable_length_batching_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise NTError(status, where, lib().nt_last_error().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return NT_BF16
    if t.dtype == torch.float32:
        return NT_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _f32(t: Optional[torch.Tensor]):
    if t is not None and t.dtype != torch.float32:
        raise ValueError("LayerNorm parameters and biases are fp32")
    return t


@dataclass
class Partition:
    """Device partitions of a packed batch plus the host totals.  For a
    rectangular batch ``col_lengths`` / ``col_cu_seqlens`` hold M_i and its
    scan; for a square one they are the row tensors."""
    lengths: torch.Tensor
    cu_seqlens: torch.Tensor
    pair_off: torch.Tensor
    totals: torch.Tensor
    row_start: torch.Tensor
    row_sample: torch.Tensor
    c: nt_partition
    col_lengths: Optional[torch.Tensor] = None
    col_cu_seqlens: Optional[torch.Tensor] = None

    @property
    def T_cols(self): return self.c.T_cols

    @property
    def max_col_len(self): return self.c.max_col_len

    @property
    def B(self): return self.c.B

    @property
    def T(self): return self.c.T

    @property
    def P(self): return self.c.P

    @property
    def max_len(self): return self.c.max_len


def nt_partition_build(lengths: torch.Tensor, stream=None, T: Optional[int] = None) -> Partition:
    """Sizes N_i (int32, on the device) -> cu_seqlens, pair offsets and the
    second-level row splits (``nt_partition_build`` + ``nt_partition_rows``).
    ``T``, when the caller knows the lengths' sum (the packed singles' row
    count), selects ``nt_partition_build_with_rows``: one host round trip."""
    if lengths.dtype != torch.int32:
        raise ValueError("lengths must be int32")
    dev = lengths.device
    B = lengths.numel()
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    pair_off = torch.empty(B + 1, dtype=torch.int64, device=dev)
    totals = torch.empty(4, dtype=torch.int64, device=dev)
    c = nt_partition()
    if T is not None:
        row_start = torch.empty(int(T) + 1, dtype=torch.int64, device=dev)
        row_sample = torch.empty(max(int(T), 1), dtype=torch.int32, device=dev)
        st = lib().nt_partition_build_with_rows(_ptr(lengths) if B else None, B, int(T), _ptr(cu), _ptr(pair_off),
                                                _ptr(totals), _ptr(row_start), _ptr(row_sample), ctypes.byref(c),
                                                _stream(stream))
        _check(st, "nt_partition_build_with_rows")
        return Partition(lengths, cu, pair_off, totals, row_start, row_sample, c)
    st = lib().nt_partition_build(_ptr(lengths) if B else None, B, _ptr(cu), _ptr(pair_off),
                                  _ptr(totals), ctypes.byref(c), _stream(stream))
    _check(st, "nt_partition_build")
    row_start = torch.empty(c.T + 1, dtype=torch.int64, device=dev)
    row_sample = torch.empty(max(c.T, 1), dtype=torch.int32, device=dev)
    _check(lib().nt_partition_rows(ctypes.byref(c), _ptr(row_start), _ptr(row_sample), _stream(stream)),
           "nt_partition_rows")
    return Partition(lengths, cu, pair_off, totals, row_start, row_sample, c)


def nt_partition_build_rect(rows: torch.Tensor, cols: torch.Tensor, stream=None) -> Partition:
    """Row lengths N_i and column lengths M_i (int32, on the device) ->
    partitions of the N_i x M_i pair states (``nt_partition_build_rect`` +
    ``nt_partition_rows``)."""
    if rows.dtype != torch.int32 or cols.dtype != torch.int32:
        raise ValueError("lengths must be int32")
    if rows.numel() != cols.numel():
        raise ValueError("one column length per sample")
    dev = rows.device
    B = rows.numel()
    cu_r = torch.empty(B + 1, dtype=torch.int32, device=dev)
    cu_c = torch.empty(B + 1, dtype=torch.int32, device=dev)
    pair_off = torch.empty(B + 1, dtype=torch.int64, device=dev)
    totals = torch.empty(8, dtype=torch.int64, device=dev)
    c = nt_partition()
    st = lib().nt_partition_build_rect(_ptr(rows) if B else None, _ptr(cols) if B else None, B, _ptr(cu_r),
                                       _ptr(cu_c), _ptr(pair_off), _ptr(totals), ctypes.byref(c), _stream(stream))
    _check(st, "nt_partition_build_rect")
    row_start = torch.empty(c.T + 1, dtype=torch.int64, device=dev)
    row_sample = torch.empty(max(c.T, 1), dtype=torch.int32, device=dev)
    _check(lib().nt_partition_rows(ctypes.byref(c), _ptr(row_start), _ptr(row_sample), _stream(stream)),
           "nt_partition_rows")
    return Partition(rows, cu_r, pair_off, totals, row_start, row_sample, c, cols, cu_c)


def nt_pair_broadcast_workspace_bytes(T: int, C_z: int) -> int:
    return int(lib().nt_pair_broadcast_workspace_bytes(T, C_z))


def nt_pair_broadcast_workspace_bytes_rect(T_rows: int, T_cols: int, C_z: int) -> int:
    return int(lib().nt_pair_broadcast_workspace_bytes_rect(T_rows, T_cols, C_z))


def nt_pair_broadcast(part: Partition, s_left: torch.Tensor, s_right: torch.Tensor,
                      W_a: torch.Tensor, W_b: torch.Tensor, z: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    T, C_s = s_left.shape
    C_z = W_a.shape[0]
    if T != part.T or tuple(s_right.shape) != (part.T_cols, C_s):
        raise ValueError(f"singles {tuple(s_left.shape)}, {tuple(s_right.shape)} do not match the partition "
                         f"(T={part.T}, T_cols={part.T_cols})")
    if tuple(W_a.shape) != (C_z, C_s) or tuple(W_b.shape) != (C_z, C_s):
        raise ValueError("W_a, W_b must be (C_z, C_s)")
    if z is None:
        z = torch.empty(part.P, C_z, dtype=s_left.dtype, device=s_left.device)
    elif tuple(z.shape) != (part.P, C_z):
        raise ValueError(f"z {tuple(z.shape)} must be (P={part.P}, C_z={C_z})")
    need = nt_pair_broadcast_workspace_bytes_rect(T, part.T_cols, C_z)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=s_left.device)
    st = lib().nt_pair_broadcast(ctypes.byref(part.c), _dtype(s_left), _ptr(s_left), _ptr(s_right), C_s,
                                 _ptr(W_a), _ptr(W_b), C_z, _ptr(z), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nt_pair_broadcast")
    return z


def nt_pair_broadcast_noalloc(part: Partition, s_left: torch.Tensor, s_right: torch.Tensor,
                              W_a: torch.Tensor, W_b: torch.Tensor, z: Optional[torch.Tensor] = None,
                              stream=None) -> torch.Tensor:
    """nt_pair_broadcast without a workspace argument: u and v live in the
    library's own fixed device array ((T + T_cols) * C_z <= 2,097,152), for callers
    that cannot allocate device memory.  ``z`` must then be supplied by the
    caller too if the call itself may not allocate."""
    T, C_s = s_left.shape
    C_z = W_a.shape[0]
    if z is None:
        z = torch.empty(part.P, C_z, dtype=s_left.dtype, device=s_left.device)
    st = lib().nt_pair_broadcast_noalloc(ctypes.byref(part.c), _dtype(s_left), _ptr(s_left), _ptr(s_right),
                                         C_s, _ptr(W_a), _ptr(W_b), C_z, _ptr(z), _stream(stream))
    _check(st, "nt_pair_broadcast_noalloc")
    return z


def nt_pair_transition(part: Partition, z: torch.Tensor, ln_gamma: torch.Tensor, ln_beta: torch.Tensor,
                       W1: torch.Tensor, b1: Optional[torch.Tensor], W2: torch.Tensor,
                       b2: Optional[torch.Tensor], ln_eps: float = 1e-5,
                       out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    P, C_z = z.shape
    H_t = W1.shape[0]
    if P != part.P:
        raise ValueError(f"z has {P} cells, the partition {part.P}")
    if tuple(W1.shape) != (H_t, C_z) or tuple(W2.shape) != (C_z, H_t):
        raise ValueError("W1 must be (H_t, C_z) and W2 (C_z, H_t)")
    if out is None:
        out = torch.empty_like(z)
    st = lib().nt_pair_transition(ctypes.byref(part.c), _dtype(z), _ptr(z), _ptr(out), C_z, H_t,
                                  _ptr(_f32(ln_gamma)), _ptr(_f32(ln_beta)), ln_eps, _ptr(W1),
                                  _ptr(_f32(b1)), _ptr(W2), _ptr(_f32(b2)), _stream(stream))
    _check(st, "nt_pair_transition")
    return out


def nt_pair_transition_swiglu(part: Partition, z: torch.Tensor, ln_gamma: torch.Tensor, ln_beta: torch.Tensor,
                              W1: torch.Tensor, b1: Optional[torch.Tensor], W3: torch.Tensor,
                              b3: Optional[torch.Tensor], W2: torch.Tensor, b2: Optional[torch.Tensor],
                              ln_eps: float = 1e-5, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """z~ = z + W2 (SiLU(W1 LN(z) + b1) * (W3 LN(z) + b3)) + b2 per cell."""
    P, C_z = z.shape
    H_t = W1.shape[0]
    if P != part.P:
        raise ValueError(f"z has {P} cells, the partition {part.P}")
    if tuple(W1.shape) != (H_t, C_z) or tuple(W3.shape) != (H_t, C_z) or tuple(W2.shape) != (C_z, H_t):
        raise ValueError("W1 and W3 must be (H_t, C_z) and W2 (C_z, H_t)")
    if out is None:
        out = torch.empty_like(z)
    st = lib().nt_pair_transition_swiglu(ctypes.byref(part.c), _dtype(z), _ptr(z), _ptr(out), C_z, H_t,
                                         _ptr(_f32(ln_gamma)), _ptr(_f32(ln_beta)), ln_eps, _ptr(W1),
                                         _ptr(_f32(b1)), _ptr(W3), _ptr(_f32(b3)), _ptr(W2), _ptr(_f32(b2)),
                                         _stream(stream))
    _check(st, "nt_pair_transition_swiglu")
    return out


def nt_pair_transition_cells(z: torch.Tensor, ln_gamma: torch.Tensor, ln_beta: torch.Tensor, W1: torch.Tensor,
                             b1: Optional[torch.Tensor], W2: torch.Tensor, b2: Optional[torch.Tensor],
                             W3: Optional[torch.Tensor] = None, b3: Optional[torch.Tensor] = None,
                             ln_eps: float = 1e-5, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The transition over the cells of ``z`` (any slice of a pair state,
    rows contiguous), with no partition: ReLU, or SwiGLU when ``W3`` is given.
    Each cell's result equals the whole-state call's bit for bit."""
    P, C_z = z.shape
    H_t = W1.shape[0]
    if tuple(W1.shape) != (H_t, C_z) or tuple(W2.shape) != (C_z, H_t) or \
            (W3 is not None and tuple(W3.shape) != (H_t, C_z)):
        raise ValueError("W1 (and W3) must be (H_t, C_z) and W2 (C_z, H_t)")
    if not z.is_contiguous():
        raise ValueError("z must be contiguous")
    if out is None:
        out = torch.empty_like(z)
    st = lib().nt_pair_transition_cells(P, _dtype(z), _ptr(z), _ptr(out), C_z, H_t, _ptr(_f32(ln_gamma)),
                                        _ptr(_f32(ln_beta)), ln_eps, _ptr(W1), _ptr(_f32(b1)), _ptr(W3),
                                        _ptr(_f32(b3)), _ptr(W2), _ptr(_f32(b2)), _stream(stream))
    _check(st, "nt_pair_transition_cells")
    return out


def nt_pair_reduce(part: Partition, z: torch.Tensor, W_g: Optional[torch.Tensor] = None,
                   b_g: Optional[torch.Tensor] = None, s_in: Optional[torch.Tensor] = None,
                   m: Optional[torch.Tensor] = None, s_out: Optional[torch.Tensor] = None,
                   stream=None):
    P, C_z = z.shape
    if P != part.P:
        raise ValueError(f"z has {P} cells, the partition {part.P}")
    if m is None:
        m = torch.empty(part.T, C_z, dtype=z.dtype, device=z.device)
    C_s = 0
    if W_g is not None:
        C_s = W_g.shape[0]
        if tuple(W_g.shape) != (C_s, C_z):
            raise ValueError("W_g must be (C_s, C_z)")
        if s_out is None:
            s_out = torch.empty(part.T, C_s, dtype=z.dtype, device=z.device)
    st = lib().nt_pair_reduce(ctypes.byref(part.c), _dtype(z), _ptr(z), C_z, _ptr(m), _ptr(W_g),
                              _ptr(_f32(b_g)), _ptr(s_in), _ptr(s_out), C_s, _stream(stream))
    _check(st, "nt_pair_reduce")
    return m, s_out


def nt_pair_reduce_loss(part: Partition, z: torch.Tensor, W_g: torch.Tensor, b_g: Optional[torch.Tensor] = None,
                        s_in: Optional[torch.Tensor] = None, m: Optional[torch.Tensor] = None,
                        s_out: Optional[torch.Tensor] = None, loss: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None):
    """The reduce with the g projection and the Eq. 5 loss of (s_out, z) in
    one call that reads z once: returns (m, s_out, loss as a 1-element fp32
    device tensor).  ``m``, ``s_out``, ``loss`` and ``workspace`` (of
    nt_pair_reduce_loss_workspace_bytes() bytes) may be given, so that a
    captured graph writes into fixed buffers."""
    P, C_z = z.shape
    if P != part.P:
        raise ValueError(f"z has {P} cells, the partition {part.P}")
    C_s = W_g.shape[0]
    if tuple(W_g.shape) != (C_s, C_z):
        raise ValueError("W_g must be (C_s, C_z)")
    dev = z.device
    if m is None:
        m = torch.empty(part.T, C_z, dtype=z.dtype, device=dev)
    if s_out is None:
        s_out = torch.empty(part.T, C_s, dtype=z.dtype, device=dev)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(int(lib().nt_pair_reduce_loss_workspace_bytes()), dtype=torch.uint8, device=dev)
    st = lib().nt_pair_reduce_loss(ctypes.byref(part.c), _dtype(z), _ptr(z), C_z, _ptr(m), _ptr(W_g),
                                   _ptr(_f32(b_g)), _ptr(s_in), _ptr(s_out), C_s, _ptr(loss), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nt_pair_reduce_loss")
    return m, s_out, loss


def nt_pair_block_loss(part: Partition, s_out: torch.Tensor, z_tilde: torch.Tensor, want_grads: bool = True,
                       stream=None, loss: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """Eq. 5 on one block's outputs: returns (loss as a 1-element fp32
    device tensor, dL/ds_out, dL/dz~) -- the gradients fp32, or None when
    ``want_grads`` is False.  ``loss`` and ``workspace`` may be given (a
    1-element fp32 tensor and nt_pair_block_loss_workspace_bytes() bytes),
    so that a captured graph writes into fixed buffers."""
    T, C_s = s_out.shape
    C_z = z_tilde.shape[1]
    if T != part.T or z_tilde.shape[0] != part.P:
        raise ValueError("outputs do not match the partition")
    dev = s_out.device
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    ds = torch.empty(T, C_s, dtype=torch.float32, device=dev) if want_grads else None
    dz = torch.empty(part.P, C_z, dtype=torch.float32, device=dev) if want_grads else None
    ws = workspace
    if ws is None:
        ws = torch.empty(int(lib().nt_pair_block_loss_workspace_bytes()), dtype=torch.uint8, device=dev)
    st = lib().nt_pair_block_loss(ctypes.byref(part.c), _dtype(s_out), _ptr(s_out), C_s, _ptr(z_tilde), C_z,
                                  _ptr(loss), _ptr(ds), _ptr(dz), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "nt_pair_block_loss")
    return loss, ds, dz


def nt_pair_block_backward(part: Partition, s: torch.Tensor, w, m: torch.Tensor, ds_out: torch.Tensor,
                           dz_tilde: Optional[torch.Tensor] = None, ln_eps: float = 1e-5, workspace=None,
                           stream=None):
    """Gradients of one block (ReLU transition) for upstream gradients of its
    outputs; ``w`` holds the forward's parameters.  Returns a dict of fp32
    tensors: ds, dW_a, dW_b, dgamma, dbeta, dW1, db1, dW2, db2, dW_g, db_g."""
    T, C_s = s.shape
    C_z = w.W_a.shape[0]
    H_t = w.W1.shape[0]
    dev = s.device
    f = lambda *shape: torch.empty(*shape, dtype=torch.float32, device=dev)
    g = {"ds": f(T, C_s), "dW_a": f(C_z, C_s), "dW_b": f(C_z, C_s), "dgamma": f(C_z), "dbeta": f(C_z),
         "dW1": f(H_t, C_z), "db1": f(H_t), "dW2": f(C_z, H_t), "db2": f(C_z), "dW_g": f(C_s, C_z), "db_g": f(C_s)}
    need = nt_pair_block_backward_workspace_bytes(_dtype(s), part.T, part.P, C_z, H_t)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = lib().nt_pair_block_backward(
        ctypes.byref(part.c), _dtype(s), _ptr(s), C_s, _ptr(w.W_a), _ptr(w.W_b), C_z, H_t, _ptr(_f32(w.ln_gamma)),
        _ptr(_f32(w.ln_beta)), float(ln_eps), _ptr(w.W1), _ptr(_f32(w.b1)), _ptr(w.W2), _ptr(w.W_g), _ptr(m),
        _ptr(ds_out), _ptr(dz_tilde), _ptr(g["ds"]), _ptr(g["dW_a"]), _ptr(g["dW_b"]), _ptr(g["dgamma"]),
        _ptr(g["dbeta"]), _ptr(g["dW1"]), _ptr(g["db1"]), _ptr(g["dW2"]), _ptr(g["db2"]), _ptr(g["dW_g"]),
        _ptr(g["db_g"]), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nt_pair_block_backward")
    return g


def nt_pair_block_loss_backward(part: Partition, s: torch.Tensor, w, m: torch.Tensor, s_out: torch.Tensor,
                                z_tilde: torch.Tensor, ln_eps: float = 1e-5, loss: Optional[torch.Tensor] = None,
                                workspace=None, stream=None):
    """Eq. 5 on the block's outputs and the block's gradients for it, in one
    call: returns (loss as a 1-element fp32 device tensor, the gradient dict
    of :func:`nt_pair_block_backward`).  Equal, value for value, to
    nt_pair_block_loss followed by nt_pair_block_backward with its gradients;
    on the tensor-core route dL/dz~ is formed from z~ where it is read."""
    T, C_s = s.shape
    C_z = w.W_a.shape[0]
    H_t = w.W1.shape[0]
    if s_out.shape[0] != part.T or z_tilde.shape[0] != part.P:
        raise ValueError("outputs do not match the partition")
    dev = s.device
    f = lambda *shape: torch.empty(*shape, dtype=torch.float32, device=dev)
    g = {"ds": f(T, C_s), "dW_a": f(C_z, C_s), "dW_b": f(C_z, C_s), "dgamma": f(C_z), "dbeta": f(C_z),
         "dW1": f(H_t, C_z), "db1": f(H_t), "dW2": f(C_z, H_t), "db2": f(C_z), "dW_g": f(C_s, C_z), "db_g": f(C_s)}
    if loss is None:
        loss = f(1)
    need = nt_pair_block_loss_backward_workspace_bytes(_dtype(s), part.T, part.P, C_s, C_z, H_t)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = lib().nt_pair_block_loss_backward(
        ctypes.byref(part.c), _dtype(s), _ptr(s), C_s, _ptr(w.W_a), _ptr(w.W_b), C_z, H_t, _ptr(_f32(w.ln_gamma)),
        _ptr(_f32(w.ln_beta)), float(ln_eps), _ptr(w.W1), _ptr(_f32(w.b1)), _ptr(w.W2), _ptr(w.W_g), _ptr(m),
        _ptr(s_out), _ptr(z_tilde), _ptr(loss), _ptr(g["ds"]), _ptr(g["dW_a"]), _ptr(g["dW_b"]), _ptr(g["dgamma"]),
        _ptr(g["dbeta"]), _ptr(g["dW1"]), _ptr(g["db1"]), _ptr(g["dW2"]), _ptr(g["db2"]), _ptr(g["dW_g"]),
        _ptr(g["db_g"]), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nt_pair_block_loss_backward")
    return loss, g


def nt_pair_block_loss_backward_workspace_bytes(dtype: int, T: int, P: int, C_s: int, C_z: int, H_t: int) -> int:
    """Device workspace bytes of nt_pair_block_loss_backward."""
    return int(lib().nt_pair_block_loss_backward_workspace_bytes(int(dtype), int(T), int(P), int(C_s), int(C_z),
                                                                 int(H_t)))


def nt_pair_block_backward_workspace_bytes(dtype: int, T: int, P: int, C_z: int, H_t: int) -> int:
    """Device workspace bytes of nt_pair_block_backward (dtype: NT_F32 / NT_BF16 code)."""
    return int(lib().nt_pair_block_backward_workspace_bytes(int(dtype), int(T), int(P), int(C_z), int(H_t)))


def nt_varlen_attn_workspace_bytes() -> int:
    return int(lib().nt_varlen_attn_workspace_bytes())


def _attn_workspace(workspace, device):
    """The attention calls' work-counter workspace: a given uint8 tensor, a
    fresh one (None), or no workspace at all (False: one CTA per item)."""
    if workspace is False:
        return None, 0
    if workspace is None:
        workspace = torch.empty(nt_varlen_attn_workspace_bytes(), dtype=torch.uint8, device=device)
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def nt_varlen_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                   max_len: int, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, want_lse: bool = False, stream=None, workspace=None):
    """``workspace``: a device tensor of at least nt_varlen_attn_workspace_bytes()
    bytes for the persistent schedule's work counter (None allocates one per
    call; False passes none, which runs one CTA per work item)."""
    T, H, d = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share the shape (T, H, d)")
    if cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    B = cu_seqlens.numel() - 1
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty(H, T, dtype=torch.float32, device=q.device)
    ws, ws_bytes = _attn_workspace(workspace, q.device)
    st = lib().nt_varlen_attn(_dtype(q), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), B, T, int(max_len),
                              H, d, float(scale), _ptr(out), _ptr(lse), ws, ws_bytes, _stream(stream))
    _check(st, "nt_varlen_attn")
    return out, lse


def nt_varlen_attn_qk(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                      cu_seqlens_k: torch.Tensor, max_len_q: int, scale: Optional[float] = None,
                      causal: bool = False, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, want_lse: bool = False, stream=None,
                      workspace=None):
    """Queries of segment b attend to keys [cu_k[b], cu_k[b+1]); with
    ``causal`` the diagonal is aligned to each segment's bottom-right corner.
    ``workspace`` as in :func:`nt_varlen_attn`."""
    T_q, H, d = q.shape
    T_k = k.shape[0]
    if tuple(k.shape[1:]) != (H, d) or v.shape != k.shape:
        raise ValueError("k and v must be (T_k, H, d) with q's H and d")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have B+1 entries each")
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if want_lse and lse is None:
        lse = torch.empty(H, T_q, dtype=torch.float32, device=q.device)
    ws, ws_bytes = _attn_workspace(workspace, q.device)
    st = lib().nt_varlen_attn_qk(_dtype(q), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                 B, T_q, T_k, int(max_len_q), H, d, float(scale), int(bool(causal)),
                                 _ptr(out), _ptr(lse), ws, ws_bytes, _stream(stream))
    _check(st, "nt_varlen_attn_qk")
    return out, lse


def nt_varlen_attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, d_o: torch.Tensor,
                       lse: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: Optional[torch.Tensor],
                       max_len_q: int, max_len_k: Optional[int] = None, scale: Optional[float] = None,
                       causal: bool = False, stream=None):
    """Gradients (dq, dk, dv) of varlen attention for the upstream gradient
    ``d_o``, from the forward's ``o`` and natural-log ``lse`` [H, T_q].
    ``cu_seqlens_k`` None means the query offsets (self-attention); the max
    lengths bound the longest segment of each side (``max_len_k`` defaults
    to ``max_len_q``)."""
    T_q, H, d = q.shape
    T_k = k.shape[0]
    if cu_seqlens_k is None:
        cu_seqlens_k = cu_seqlens_q
    if max_len_k is None:
        max_len_k = max_len_q
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, T_q):
        raise ValueError("lse must be fp32 (H, T_q)")
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = d ** -0.5
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(int(lib().nt_varlen_attn_bwd_workspace_bytes(T_q, H)), 16), dtype=torch.uint8,
                     device=q.device)
    st = lib().nt_varlen_attn_bwd(_dtype(q), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(d_o), _ptr(lse),
                                  _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, T_q, T_k, int(max_len_q),
                                  int(max_len_k), H, d, float(scale),
                                  int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                  ws.numel(), _stream(stream))
    _check(st, "nt_varlen_attn_bwd")
    return dq, dk, dv


def nt_device_status(stream=None) -> int:
    """Synchronise and return (then clear) the device status word as a
    status code; raises on a timeout or failed device check."""
    st = lib().nt_device_status(_stream(stream))
    _check(st, "nt_device_status")
    return st


def nt_selftest_bounded_wait(mode: int, delay_ns: int, limit_ns: int, result: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """The device-side wait self-test (mode 0: completed after ``delay_ns``;
    1: runs out after ``limit_ns`` and flags a timeout; 2: given up on the
    CTA's abort flag after ``delay_ns``).  Returns the int64[2] device tensor
    (succeeded, duration in ns) it writes asynchronously; nt_device_status
    then reports what was flagged."""
    if result is None:
        result = torch.full((2,), -1, dtype=torch.int64, device="cuda")
    st = lib().nt_selftest_bounded_wait(int(mode), int(delay_ns), int(limit_ns), _ptr(result), _stream(stream))
    _check(st, "nt_selftest_bounded_wait")
    return result


def nt_pair_block_fused(part: Partition, s_left: torch.Tensor, s_right: torch.Tensor, w, W3=None, b3=None,
                        ln_eps: float = 1e-5, z: Optional[torch.Tensor] = None, m: Optional[torch.Tensor] = None,
                        s_out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None):
    """The whole block in one pass (``nt_pair_block_fused``).  ``w`` holds
    W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, b2, W_g, b_g on the device;
    ``W3`` (and ``b3``) select the SwiGLU update.  Returns (z~, m, s_out)."""
    T, C_s = s_left.shape
    C_z, H_t = w.W_a.shape[0], w.W1.shape[0]
    if T != part.T or tuple(s_right.shape) != (part.T_cols, C_s):
        raise ValueError("singles do not match the partition")
    dev, dt = s_left.device, s_left.dtype
    if z is None:
        z = torch.empty(part.P, C_z, dtype=dt, device=dev)
    if m is None:
        m = torch.empty(T, C_z, dtype=dt, device=dev)
    if s_out is None and w.W_g is not None:
        s_out = torch.empty(T, C_s, dtype=dt, device=dev)
    need = int(lib().nt_pair_block_fused_workspace_bytes(T, part.T_cols, C_z))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    st = lib().nt_pair_block_fused(
        ctypes.byref(part.c), _dtype(s_left), _ptr(s_left), _ptr(s_right), C_s, _ptr(w.W_a), _ptr(w.W_b), C_z, H_t,
        _ptr(_f32(w.ln_gamma)), _ptr(_f32(w.ln_beta)), ln_eps, _ptr(w.W1), _ptr(_f32(w.b1)), _ptr(W3), _ptr(_f32(b3)),
        _ptr(w.W2), _ptr(_f32(w.b2)), _ptr(w.W_g), _ptr(_f32(w.b_g)), _ptr(z), _ptr(m), _ptr(s_out),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "nt_pair_block_fused")
    return z, m, s_out


def block_forward(part: Partition, s: torch.Tensor, w, ln_eps: float = 1e-5,
                  z: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  s_out: Optional[torch.Tensor] = None, stream=None, s_col: Optional[torch.Tensor] = None):
    """One single->pair->single block (Eq. 1) as the three pair calls; ``w``
    holds W_a, W_b, ln_gamma, ln_beta, W1, b1, W2, b2, W_g, b_g on the device.
    The transition runs in place on z.  ``s_col`` gives the column singles of
    a rectangular partition (default: ``s``).  Returns (z~, m, s_out)."""
    z = nt_pair_broadcast(part, s, s if s_col is None else s_col, w.W_a, w.W_b, z=z, workspace=workspace,
                          stream=stream)
    nt_pair_transition(part, z, w.ln_gamma, w.ln_beta, w.W1, w.b1, w.W2, w.b2, ln_eps=ln_eps,
                       out=z, stream=stream)
    m, s_out = nt_pair_reduce(part, z, w.W_g, w.b_g, s_in=s, s_out=s_out, stream=stream)
    return z, m, s_out
