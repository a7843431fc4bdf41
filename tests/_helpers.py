"""Shared test helpers: conversion of seeded inputs to oracle float64 arrays
and the error metrics the parity tests use."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from variable_length_batching_gb300.workloads import BlockWeights, io_bits_to_f64
from oracle.block import Weights

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# Normwise tolerances: max|gpu - oracle| / max|oracle| per output tensor.
TOL = {"bf16": 2e-2, "f32": 1e-5}


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f64(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return io_bits_to_f64(t)


def oracle_weights(w: BlockWeights, eps: float = 1e-5) -> Weights:
    return Weights(W_a=f64(w.W_a), W_b=f64(w.W_b), gamma=f64(w.ln_gamma), beta=f64(w.ln_beta),
                   eps=eps, W1=f64(w.W1), b1=f64(w.b1), W2=f64(w.W2), b2=f64(w.b2),
                   W_g=f64(w.W_g), b_g=f64(w.b_g))


def normwise_err(got, ref) -> float:
    got = f64(got) if not isinstance(got, np.ndarray) else got.astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    denom = np.abs(ref).max()
    if denom == 0:
        return float(np.abs(got - ref).max())
    return float(np.abs(got - ref).max() / denom)


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()
