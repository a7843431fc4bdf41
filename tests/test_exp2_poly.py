"""The FMA-pipe exp2 of the attention kernel, derived in
variable_length_batching_gb300/exp2_poly.py, against numpy's exp2."""
import numpy as np
import pytest

pytest.importorskip("scipy")

from variable_length_batching_gb300 import exp2_poly


def test_fit_is_minimax_quality():
    c, err = exp2_poly.fit()
    assert c[0] == 1.0 and err < 1.2e-4
    # the constants compiled into the attention kernel
    assert np.allclose(c.astype(np.float32), [1.0, 0.6932829022407532, 0.2422109693288803, 0.055009059607982635],
                       rtol=0, atol=2e-7)


def test_reduced_exp2_over_range():
    c, _ = exp2_poly.fit()
    x = np.linspace(-125.0, 8.0, 400001).astype(np.float32)
    got = exp2_poly.exp2_reduced(x, c).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.abs(got / ref - 1).max() < 1.2e-4
    ints = np.arange(-120, 9).astype(np.float32)
    assert np.array_equal(exp2_poly.exp2_reduced(ints, c), np.exp2(ints))
