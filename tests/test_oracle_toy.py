"""Pins of the toy-decoder oracle's building blocks against closed forms:
the rotary embedding is the identity at position 0, preserves each rotated
pair's norm, and makes q.k depend only on the position difference; RMSNorm
with unit weight yields unit root-mean-square; SwiGLU of a zero gate is 0."""
import numpy as np

from oracle import toy_model as T


def test_rope_identity_at_zero_and_norm_preserving():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 128))
    assert np.allclose(T.rope(x, np.zeros(5), 128), x, rtol=0, atol=0)
    y = T.rope(x, np.arange(5, dtype=float) * 1000.0, 128)
    n_x = x[..., :64] ** 2 + x[..., 64:] ** 2
    n_y = y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.allclose(n_x, n_y, rtol=1e-12, atol=1e-12)


def test_rope_dot_product_depends_on_relative_position_only():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((1, 1, 128)), rng.standard_normal((1, 1, 128))
    dots = []
    for p in (0.0, 7.0, 12345.0):
        qr = T.rope(q, np.array([p + 30.0]), 128)
        kr = T.rope(k, np.array([p]), 128)
        dots.append(float((qr * kr).sum()))
    assert np.allclose(dots, dots[0], rtol=1e-9, atol=1e-9)


def test_rmsnorm_unit_rms_and_swiglu_zero_gate():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 1024)) * 7
    y = T.rmsnorm(x, np.ones(1024))
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-6)
    g = np.zeros(8)
    assert np.all(g / (1.0 + np.exp(-g)) * np.arange(8) == 0)
