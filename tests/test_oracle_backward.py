"""Pins of the oracle's Eq. 5 loss and block gradients (CPU): hand-evaluated
sample weights, closed forms of the loss, torch autograd of an independent
formulation, and central differences."""
import numpy as np

import _pins as pins
from oracle import block as oblock
from oracle import block_backward as obwd


def test_eq5_weights():
    pins.pin_eq5_weights(obwd.eq5_sample_weights)


def test_eq5_closed_form():
    pins.pin_eq5_closed_form(obwd.eq5_loss)


def test_block_backward_autograd():
    pins.pin_block_backward_autograd(obwd.block_loss_and_grads, oblock.block_packed, np.random.default_rng(5))


def test_block_backward_finite_differences():
    pins.pin_block_backward_finite_differences(obwd.block_loss_and_grads, oblock.block_packed,
                                               np.random.default_rng(6))


def test_eq5_grads_scale_outputs():
    """dL/dX~ and dL/dP~ are the outputs scaled per sample (Eq. 5 is a
    weighted sum of squares)."""
    lengths = [2, 1, 3]
    s_out = np.arange(6 * 5, dtype=np.float64).reshape(6, 5) / 7
    z = np.arange(14 * 3, dtype=np.float64).reshape(14, 3) / 11
    ds, dz = obwd.eq5_loss_grads(lengths, s_out, z)
    a, b = obwd.eq5_sample_weights(3)
    assert np.allclose(ds[0:2], 2 * a[0] * s_out[0:2] / (5 * 6))
    assert np.allclose(ds[3:6], 2 * a[2] * s_out[3:6] / (5 * 6))
    assert np.allclose(dz[4:5], 2 * b[1] * z[4:5] / (3 * 14))
