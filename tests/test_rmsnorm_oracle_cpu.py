"""Pins for oracle/rmsnorm.py: closed forms on constant rows, scale
invariance with eps = 0, the sign rule, and a one-element row."""
import numpy as np

from oracle import oracle as orc
from oracle import rmsnorm


def test_constant_row_closed_form():
    H, c, eps = 64, 3.0, 0.0
    X = np.full((1, H), c, np.float32)
    w = np.linspace(-2, 2, H).astype(np.float32)
    r, y, _ = rmsnorm.rmsnorm(X, w, eps)
    assert r[0] == 1.0 / 3.0                        # sqrt(mean(c^2)) = |c|
    assert np.allclose(y[0], w.astype(np.float64), rtol=0, atol=1e-15)


def test_eps_enters_under_the_root():
    H = 16
    X = np.full((1, H), 2.0, np.float32)
    r, _, _ = rmsnorm.rmsnorm(X, np.ones(H, np.float32), 5.0)
    assert r[0] == 1.0 / 3.0                        # 1 / sqrt(4 + 5)


def test_scale_invariance_and_sign():
    g = np.random.default_rng(0)
    X = g.standard_normal((5, 96)).astype(np.float32)
    w = g.standard_normal(96).astype(np.float32)
    _, y1, b1 = rmsnorm.rmsnorm(X, w, 0.0)
    _, y2, b2 = rmsnorm.rmsnorm(X * 4.0, w, 0.0)     # exact power-of-two scaling
    assert np.array_equal(b1, b2)
    _, y3, _ = rmsnorm.rmsnorm(-X, w, 0.0)
    assert np.array_equal(y3, -y1)


def test_one_element_row_and_bf16_inputs():
    _, y, b = rmsnorm.rmsnorm(np.array([[-7.0]], np.float32), np.array([0.5], np.float32), 0.0)
    assert y[0, 0] == -0.5 and b[0, 0] == orc.round_bf16(np.array([-0.5]))[0]
    Xb = np.array([[0x3F80, 0xC000]], np.uint16)     # bf16 1.0 and -2.0
    r, y, _ = rmsnorm.rmsnorm(Xb, np.array([0x3F80, 0x3F80], np.uint16), 0.0)
    assert np.isclose(r[0], 1.0 / np.sqrt(2.5)) and np.allclose(y[0], np.array([1.0, -2.0]) * r[0])
