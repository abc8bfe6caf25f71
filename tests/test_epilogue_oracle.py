"""Pins of the gated RMSNorm oracle (oracle/epilogue.py): closed forms of single rows, invariances
of the normalisation, and the gate's limits."""
import math

import numpy as np

import oracle.epilogue as oe


def test_one_hot_row_closed_form():
    D, a, eps = 128, 3.0, 1e-6
    x = np.zeros((1, D))
    x[0, 5] = a
    z = np.full((1, D), 2.0)
    w = np.linspace(0.5, 1.5, D)
    out = oe.gated_rms(x, z, w, eps)
    silu2 = 2.0 / (1.0 + math.exp(-2.0))
    assert math.isclose(out[0, 5], w[5] * a / math.sqrt(a * a / D + eps) * silu2, rel_tol=1e-14)
    assert np.all(out[0, np.arange(D) != 5] == 0.0)


def test_zero_gate_gives_zero_and_gate_limits():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 128))
    w = rng.uniform(0.5, 1.5, 128)
    assert np.all(oe.gated_rms(x, np.zeros((3, 128)), w) == 0.0)
    big = oe.gated_rms(x, np.full((3, 128), 40.0), w)          # silu(z) -> z for large z
    ref = w * x / np.sqrt(np.mean(x * x, -1, keepdims=True) + 1e-6) * 40.0
    assert np.allclose(big, ref, rtol=1e-15)
    neg = oe.gated_rms(x, np.full((3, 128), -40.0), w)         # silu(z) -> z e^z for very negative z
    assert np.all(np.abs(neg) < 1e-14)


def test_scale_invariance_without_eps_and_linearity_in_w():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 128))
    z = rng.standard_normal((4, 128))
    w = rng.uniform(0.5, 1.5, 128)
    assert np.allclose(oe.gated_rms(7.5 * x, z, w, 0.0), oe.gated_rms(x, z, w, 0.0), rtol=1e-14)
    assert np.allclose(oe.gated_rms(x, z, 2 * w), 2 * oe.gated_rms(x, z, w), rtol=1e-15)
    # each row is normalised by its own mean square: the row means of x_hat^2 are 1 (eps = 0)
    xh = oe.gated_rms(x, np.full_like(z, 40.0), np.ones(128), 0.0) / 40.0
    assert np.allclose(np.mean(xh * xh, -1), 1.0, rtol=1e-14)


def test_rows_are_independent():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 128))
    z = rng.standard_normal((5, 128))
    w = rng.uniform(0.5, 1.5, 128)
    full = oe.gated_rms(x, z, w)
    for i in range(5):
        assert np.array_equal(oe.gated_rms(x[i:i + 1], z[i:i + 1], w), full[i:i + 1])
