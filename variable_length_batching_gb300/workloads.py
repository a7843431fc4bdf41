"""Seeded synthetic workloads for the packed single->pair->single block and
for variable-length attention.

This module only draws numbers: per-sample lengths, single representations,
weights and Q/K/V, cast to the I/O dtype.  It holds none of the method's
arithmetic (no offsets, no projections, no reductions), so both the CUDA path
and the CPU oracle can take their inputs from here without sharing any code
that computes the block.

Shapes and distributions follow the workloads of "DanLing NestedTensor:
Composable Multi-Ragged Tensors for Deep Learning" (section 4.3: B=8, single
width 384, pair width 128, transition expansion four; Appendix A.1) and the
packed-stream attention of "Variable-length attention and data packing"
(section "Core math": padding-rate model).  No dataset is used anywhere.

Every generator uses ``numpy.random.default_rng(seed)`` and draws in a fixed
order: lengths, singles, then per block W_a, W_b, W1, W2, W_g; for attention
lengths, then q, k, v.  Weights follow the paper's Linear convention
``y = x W^T + b`` (section 3.3, "Dense work across valid positions"), so every
weight is stored (out_features, in_features), row-major.  "N(0, 1/fan_in)"
is read as variance 1/fan_in.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

F32 = "f32"
BF16 = "bf16"

TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


@dataclass(frozen=True)
class BlockConfig:
    """One single->pair->single workload.

    ``lengths`` is either a fixed tuple or a rule name understood by
    :func:`draw_lengths`.
    """

    name: str
    B: int
    length_rule: str
    C_s: int
    C_z: int
    H_t: int
    dtype: str
    n_blocks: int = 1
    seed: int = 0
    fixed_lengths: Optional[Sequence[int]] = None
    rule_args: tuple = ()
    ln_eps: float = 1e-5


@dataclass(frozen=True)
class AttnConfig:
    """One packed-stream varlen attention workload."""

    name: str
    total_tokens: int
    len_lo: int
    len_hi: int
    H: int
    d: int
    dtype: str = BF16
    seed: int = 0


# The five workloads.  Sizes quoted in comments are what seed 0 draws.
TINY_FP32 = BlockConfig(  # B=4 -> T=86, P=1,966
    "tiny_fp32_B4_N8-32_Cs32_Cz16", B=4, length_rule="uniform", rule_args=(8, 32),
    C_s=32, C_z=16, H_t=64, dtype=F32)
PAIRFORMER_BF16 = BlockConfig(  # T=1,031, P=157,023
    "pairformer_bf16_B8_N64-256_Cs384_Cz128", B=8, length_rule="uniform",
    rule_args=(64, 256), C_s=384, C_z=128, H_t=512, dtype=BF16)
LOGNORMAL_BF16 = BlockConfig(  # T=3,245, P=956,323
    "lognormal_bf16_B16_mu200_s0.8_Cs384_Cz128", B=16, length_rule="lognormal",
    rule_args=(200.0, 0.8, 32, 768), C_s=384, C_z=128, H_t=512, dtype=BF16)
NEAR_UNIFORM_BF16 = BlockConfig(  # T=11,748, P=8,633,186
    "near_uniform_bf16_B16_N700-768_Cs384_Cz128", B=16, length_rule="uniform",
    rule_args=(700, 768), C_s=384, C_z=128, H_t=512, dtype=BF16)
STACKED4_BF16 = BlockConfig(  # T=3,328, P=2,170,880
    "stacked4_bf16_B8_skewed1024-64_Cs384_Cz128", B=8, length_rule="fixed",
    fixed_lengths=(1024, 768, 512, 384, 256, 192, 128, 64),
    C_s=384, C_z=128, H_t=512, dtype=BF16, n_blocks=4)
VARLEN_ATTN_BF16 = AttnConfig(  # 237 segments, sum n^2 = 23,342,596
    "varlen_attn_bf16_T65536_N16-512_H12_d64", total_tokens=65536, len_lo=16,
    len_hi=512, H=12, d=64)

BLOCK_CONFIGS = {c.name: c for c in
                 (TINY_FP32, PAIRFORMER_BF16, LOGNORMAL_BF16, NEAR_UNIFORM_BF16,
                  STACKED4_BF16)}

# Equivalent padding rates of the attention sweep (fractions).
PADDING_SWEEP = (0.03, 0.10, 0.25, 0.48, 0.75, 0.90)
PAD_TO = 512


def draw_lengths(cfg: BlockConfig, rng: np.random.Generator) -> np.ndarray:
    """Per-sample lengths N_b as int32, drawn first from ``rng``."""
    if cfg.length_rule == "fixed":
        return np.asarray(cfg.fixed_lengths, dtype=np.int32)
    if cfg.length_rule == "uniform":
        lo, hi = cfg.rule_args
        return rng.integers(lo, hi + 1, size=cfg.B).astype(np.int32)
    if cfg.length_rule == "lognormal":
        median, sigma, lo, hi = cfg.rule_args
        x = rng.lognormal(np.log(median), sigma, size=cfg.B)
        return np.clip(np.round(x), lo, hi).astype(np.int32)
    raise ValueError(f"unknown length rule {cfg.length_rule!r}")


def _normal(rng, shape, var):
    return (rng.standard_normal(shape) * np.sqrt(var)).astype(np.float32)


def to_io(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Host tensor in the I/O dtype (round-to-nearest-even for bf16)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(TORCH_DTYPE[dtype])


@dataclass
class BlockWeights:
    W_a: torch.Tensor      # (C_z, C_s)
    W_b: torch.Tensor      # (C_z, C_s)
    ln_gamma: torch.Tensor  # (C_z,) fp32
    ln_beta: torch.Tensor   # (C_z,) fp32
    W1: torch.Tensor       # (H_t, C_z)
    b1: Optional[torch.Tensor]  # (H_t,) fp32 or None
    W2: torch.Tensor       # (C_z, H_t)
    b2: Optional[torch.Tensor]  # (C_z,) fp32 or None
    W_g: torch.Tensor      # (C_s, C_z)
    b_g: Optional[torch.Tensor]  # (C_s,) fp32 or None


@dataclass
class SwiGLUWeights:
    """The SwiGLU transition's parameters: gate W1 and value W3 (H_t, C_z),
    output W2 (C_z, H_t), LN gamma/beta and optional fp32 biases."""
    ln_gamma: torch.Tensor
    ln_beta: torch.Tensor
    W1: torch.Tensor
    b1: Optional[torch.Tensor]
    W3: torch.Tensor
    b3: Optional[torch.Tensor]
    W2: torch.Tensor
    b2: Optional[torch.Tensor]


def make_swiglu_weights(C_z: int, H_t: int, dtype: str, biases: bool = False, seed: int = 0) -> SwiGLUWeights:
    """N(0, 1/fan_in) weights drawn in the order W1, W3, W2 (then biases,
    gamma, beta when ``biases``)."""
    rng = np.random.default_rng(seed)
    W1 = to_io(_normal(rng, (H_t, C_z), 1.0 / C_z), dtype)
    W3 = to_io(_normal(rng, (H_t, C_z), 1.0 / C_z), dtype)
    W2 = to_io(_normal(rng, (C_z, H_t), 1.0 / H_t), dtype)
    if biases:
        b1 = torch.from_numpy(_normal(rng, (H_t,), 0.25))
        b3 = torch.from_numpy(_normal(rng, (H_t,), 0.25))
        b2 = torch.from_numpy(_normal(rng, (C_z,), 0.25))
        gamma = torch.from_numpy(1.0 + _normal(rng, (C_z,), 0.04))
        beta = torch.from_numpy(_normal(rng, (C_z,), 0.04))
    else:
        b1 = b3 = b2 = None
        gamma = torch.ones(C_z, dtype=torch.float32)
        beta = torch.zeros(C_z, dtype=torch.float32)
    return SwiGLUWeights(gamma, beta, W1, b1, W3, b3, W2, b2)


@dataclass
class BlockInputs:
    cfg: BlockConfig
    lengths: np.ndarray            # int32 (B,)
    s: torch.Tensor                # (T, C_s) in the I/O dtype, host
    blocks: List[BlockWeights] = field(default_factory=list)


def make_block_weights(rng, C_s, C_z, H_t, dtype, biases=False) -> BlockWeights:
    W_a = to_io(_normal(rng, (C_z, C_s), 1.0 / C_s), dtype)
    W_b = to_io(_normal(rng, (C_z, C_s), 1.0 / C_s), dtype)
    W1 = to_io(_normal(rng, (H_t, C_z), 1.0 / C_z), dtype)
    W2 = to_io(_normal(rng, (C_z, H_t), 1.0 / H_t), dtype)
    W_g = to_io(_normal(rng, (C_s, C_z), 1.0 / C_z), dtype)
    if biases:
        b1 = torch.from_numpy(_normal(rng, (H_t,), 0.25))
        b2 = torch.from_numpy(_normal(rng, (C_z,), 0.25))
        b_g = torch.from_numpy(_normal(rng, (C_s,), 0.25))
        gamma = torch.from_numpy(1.0 + _normal(rng, (C_z,), 0.04))
        beta = torch.from_numpy(_normal(rng, (C_z,), 0.04))
    else:
        b1 = b2 = b_g = None
        gamma = torch.ones(C_z, dtype=torch.float32)
        beta = torch.zeros(C_z, dtype=torch.float32)
    return BlockWeights(W_a, W_b, gamma, beta, W1, b1, W2, b2, W_g, b_g)


def make_block_inputs(cfg: BlockConfig, lengths: Optional[Sequence[int]] = None,
                      biases: bool = False, seed: Optional[int] = None) -> BlockInputs:
    """Seeded inputs for ``cfg``; ``lengths`` overrides the drawn lengths."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    drawn = draw_lengths(cfg, rng)
    lens = drawn if lengths is None else np.asarray(lengths, dtype=np.int32)
    T = int(lens.astype(np.int64).sum())
    s = to_io(rng.standard_normal((T, cfg.C_s)).astype(np.float32), cfg.dtype)
    blocks = [make_block_weights(rng, cfg.C_s, cfg.C_z, cfg.H_t, cfg.dtype, biases)
              for _ in range(cfg.n_blocks)]
    return BlockInputs(cfg, lens, s, blocks)


# Rectangular pair states: the Pairformer-style block with independent row
# and column lengths, both ~ U[64, 256], rows drawn first.
RECT_BF16 = BlockConfig(  # T_rows=1,031, T_cols=1,543, P=187,394
    "rect_bf16_B8_N64-256xM64-256_Cs384_Cz128", B=8, length_rule="uniform",
    rule_args=(64, 256), C_s=384, C_z=128, H_t=512, dtype=BF16)
RECT_TINY_FP32 = BlockConfig(
    "rect_tiny_fp32_B4_N8-32xM8-32_Cs32_Cz16", B=4, length_rule="uniform", rule_args=(8, 32),
    C_s=32, C_z=16, H_t=64, dtype=F32)


@dataclass
class RectInputs:
    cfg: BlockConfig
    rows: np.ndarray      # N_i int32 (B,)
    cols: np.ndarray      # M_i int32 (B,)
    s_row: torch.Tensor   # (sum N_i, C_s) host, I/O dtype
    s_col: torch.Tensor   # (sum M_i, C_s)
    blocks: List[BlockWeights] = field(default_factory=list)


def make_rect_inputs(cfg: BlockConfig, rows: Optional[Sequence[int]] = None, cols: Optional[Sequence[int]] = None,
                     biases: bool = False, seed: Optional[int] = None) -> RectInputs:
    """Seeded rectangular inputs: row lengths, column lengths (both by the
    config's rule unless given), row singles, column singles, weights."""
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    r_drawn = draw_lengths(cfg, rng)
    c_drawn = draw_lengths(cfg, rng)
    N = r_drawn if rows is None else np.asarray(rows, dtype=np.int32)
    M = c_drawn if cols is None else np.asarray(cols, dtype=np.int32)
    s_row = to_io(rng.standard_normal((int(N.astype(np.int64).sum()), cfg.C_s)).astype(np.float32), cfg.dtype)
    s_col = to_io(rng.standard_normal((int(M.astype(np.int64).sum()), cfg.C_s)).astype(np.float32), cfg.dtype)
    blocks = [make_block_weights(rng, cfg.C_s, cfg.C_z, cfg.H_t, cfg.dtype, biases) for _ in range(cfg.n_blocks)]
    return RectInputs(cfg, N, M, s_row, s_col, blocks)


def random_rows(rows: int, width: int, dtype: str, seed: int, scale: float = 1.0) -> torch.Tensor:
    """A (rows, width) host tensor of N(0, scale^2) values in the I/O dtype."""
    rng = np.random.default_rng(seed)
    return to_io((rng.standard_normal((rows, width)) * scale).astype(np.float32), dtype)


# ----------------------------------------------------------------------------
# Attention workloads
# ----------------------------------------------------------------------------

def draw_segments(total_tokens: int, lo: int, hi: int, rng: np.random.Generator) -> np.ndarray:
    """Segment lengths drawn uniformly in [lo, hi] until they cover
    ``total_tokens``; the last segment is cut to fit."""
    out = []
    covered = 0
    while covered < total_tokens:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total_tokens - covered)
        out.append(n)
        covered += n
    return np.asarray(out, dtype=np.int32)


def sweep_length_range(rate: float, pad_to: int = PAD_TO, lo_min: int = 16):
    """Uniform length range whose mean is (1-rate)*pad_to, the expected length
    at equivalent padding ``rate`` against segments padded to ``pad_to``."""
    m = (1.0 - rate) * pad_to
    if m >= (pad_to + lo_min) / 2:
        lo, hi = int(round(2 * m - pad_to)), pad_to
    else:
        lo, hi = lo_min, int(round(2 * m - lo_min))
    return max(lo, 1), max(hi, max(lo, 1))


@dataclass
class AttnInputs:
    cfg: AttnConfig
    seqlens: np.ndarray   # int32 (B,)
    q: torch.Tensor       # (T, H, d) host, I/O dtype
    k: torch.Tensor
    v: torch.Tensor


def make_attn_inputs(cfg: AttnConfig, seqlens: Optional[Sequence[int]] = None,
                     seed: Optional[int] = None) -> AttnInputs:
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    if seqlens is None:
        lens = draw_segments(cfg.total_tokens, cfg.len_lo, cfg.len_hi, rng)
    else:
        lens = np.asarray(seqlens, dtype=np.int32)
    T = int(lens.astype(np.int64).sum())
    q = to_io(rng.standard_normal((T, cfg.H, cfg.d)).astype(np.float32), cfg.dtype)
    k = to_io(rng.standard_normal((T, cfg.H, cfg.d)).astype(np.float32), cfg.dtype)
    v = to_io(rng.standard_normal((T, cfg.H, cfg.d)).astype(np.float32), cfg.dtype)
    return AttnInputs(cfg, lens, q, k, v)


@dataclass
class CrossAttnInputs:
    seqlens_q: np.ndarray   # int32 (B,)
    seqlens_k: np.ndarray   # int32 (B,)
    q: torch.Tensor         # (T_q, H, d) host, I/O dtype
    k: torch.Tensor         # (T_k, H, d)
    v: torch.Tensor


def make_cross_attn_inputs(seqlens_q: Sequence[int], seqlens_k: Sequence[int], H: int, d: int,
                           dtype: str = BF16, seed: int = 0) -> CrossAttnInputs:
    """Queries and keys with their own per-segment lengths, N(0, 1) entries."""
    rng = np.random.default_rng(seed)
    lq = np.asarray(seqlens_q, dtype=np.int32)
    lk = np.asarray(seqlens_k, dtype=np.int32)
    if lq.shape != lk.shape:
        raise ValueError("one key length per query segment")
    Tq, Tk = int(lq.astype(np.int64).sum()), int(lk.astype(np.int64).sum())
    q = to_io(rng.standard_normal((Tq, H, d)).astype(np.float32), dtype)
    k = to_io(rng.standard_normal((Tk, H, d)).astype(np.float32), dtype)
    v = to_io(rng.standard_normal((Tk, H, d)).astype(np.float32), dtype)
    return CrossAttnInputs(lq, lk, q, k, v)


def io_bits_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a host tensor in either I/O dtype."""
    return t.detach().to("cpu").to(torch.float64).numpy()
