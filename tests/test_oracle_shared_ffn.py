"""Pins of the oracle's shared expert (oracle.shared_ffn): the expert that
"【#2】ds4.c 해독하기" keeps unquantised beside the routed experts; reading:
bf16 weights, SwiGLU with h rounded to bf16, added with weight one.

Pinned by a hand-derived two-token layer (tests/golden/shared_ffn.txt), the
closed form for constant matrices, exact linearity in w2 and in the base,
token-permutation equivariance, hidden-unit permutation invariance, and the
degenerate width 0.
"""
import numpy as np
import pytest

import oracle
from tests.golden_io import load


def _bf16(v):
    """fp32 -> bf16 bit patterns for values that are exact in bf16 (asserted)."""
    u = np.asarray(v, np.float32).view(np.uint32)
    assert not (u & 0xFFFF).any(), "test values must be exact in bf16"
    return (u >> 16).astype(np.uint16)


def _hex16(s):
    return np.array([int(t, 16) for t in s.split()], np.uint16)


def _widen(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def test_hand_computed_layer():
    g = load("shared_ffn.txt")
    w1 = _hex16(g["w1"]).reshape(2, 2)
    w3 = _hex16(g["w3"]).reshape(2, 2)
    w2 = _hex16(g["w2"]).reshape(2, 2)
    x = _hex16(g["x"]).reshape(2, 2)
    out = oracle.shared_ffn(w1, w3, w2, x)
    assert out.ravel().tolist() == [float(v) for v in g["out"].split()]
    base = np.full((2, 2), 0.5, np.float32)
    out_b = oracle.shared_ffn(w1, w3, w2, x, base)
    assert out_b.ravel().tolist() == [float(v) for v in g["out_base_half"].split()]


@pytest.mark.parametrize("a,b,c", [(0.0078125, 0.5, 0.25), (-0.015625, 0.125, 1.0)])
def test_constant_matrices_closed_form(a, b, c):
    """w1 = a, w3 = b, w2 = c everywhere: g = a sum(x), u = b sum(x), every
    hidden value is h = bf16(silu(g) u) and every output c * Fs * h."""
    rng = np.random.default_rng(3)
    D, Fs, T = 64, 48, 3
    # x with a narrow exponent range: sum(x) is exact in double
    x = _bf16(rng.integers(-64, 65, size=(T, D)) / 32.0)
    w1 = np.full((Fs, D), _bf16(a), np.uint16)
    w3 = np.full((Fs, D), _bf16(b), np.uint16)
    w2 = np.full((D, Fs), _bf16(c), np.uint16)
    out = oracle.shared_ffn(w1, w3, w2, x)
    for t in range(T):
        s = float(_widen(x[t]).astype(np.float64).sum())
        gg, uu = a * s, b * s
        hv = gg / (1.0 + np.exp(-gg)) * uu
        h = float(_widen(oracle.round_bf16(np.array([hv]))[0]))
        assert np.all(out[t] == np.float32(c * Fs * h))


def test_linear_in_w2_and_base():
    rng = np.random.default_rng(4)
    D, Fs, T = 96, 40, 4
    x = _bf16(rng.integers(-8, 9, size=(T, D)) / 8.0)
    w1 = _bf16(rng.integers(-16, 17, size=(Fs, D)) / 256.0)
    w3 = _bf16(rng.integers(-16, 17, size=(Fs, D)) / 256.0)
    w2 = _bf16(rng.integers(-16, 17, size=(D, Fs)) / 256.0)
    y = oracle.shared_ffn(w1, w3, w2, x)
    w2x2 = _bf16(2.0 * _widen(w2))
    assert np.array_equal(oracle.shared_ffn(w1, w3, w2x2, x), 2 * y)  # powers of two scale exactly
    base = rng.standard_normal((T, D)).astype(np.float32)
    got = oracle.shared_ffn(w1, w3, w2, x, base).astype(np.float64)
    # got = fp32(base + y_exact) and y = fp32(y_exact): the two differ from
    # base + y by at most half an ulp of got plus half an ulp of y
    ref = base.astype(np.float64) + y.astype(np.float64)
    bound = 0.5 * np.spacing(np.abs(got).astype(np.float32)) + 0.5 * np.spacing(np.abs(y))
    assert np.all(np.abs(got - ref) <= bound)
    assert not np.array_equal(got, y.astype(np.float64))  # the base is really added


def test_token_and_hidden_permutations():
    rng = np.random.default_rng(5)
    D, Fs, T = 80, 24, 6
    x = _bf16(rng.integers(-8, 9, size=(T, D)) / 8.0)
    w1 = _bf16(rng.integers(-16, 17, size=(Fs, D)) / 256.0)
    w3 = _bf16(rng.integers(-16, 17, size=(Fs, D)) / 256.0)
    w2 = _bf16(rng.integers(-16, 17, size=(D, Fs)) / 256.0)
    out = oracle.shared_ffn(w1, w3, w2, x)
    pt = rng.permutation(T)
    assert np.array_equal(oracle.shared_ffn(w1, w3, w2, x[pt]), out[pt])
    # permuting the hidden units (rows of w1, w3 and columns of w2 together)
    # changes only the order of the down sum: equal within its rounding
    ph = rng.permutation(Fs)
    got = oracle.shared_ffn(w1[ph], w3[ph], w2[:, ph], x)
    assert np.allclose(got, out, rtol=1e-6, atol=1e-7)
    # swapping gate and up changes the result (the SwiGLU is not symmetric)
    assert not np.array_equal(oracle.shared_ffn(w3, w1, w2, x), out)


def test_width_zero_and_argument_checks():
    x = _bf16(np.ones((2, 8), np.float32))
    z = np.zeros((0, 8), np.uint16)
    out = oracle.shared_ffn(z, z, np.zeros((8, 0), np.uint16), x)
    assert np.array_equal(out, np.zeros((2, 8), np.float32))
    base = np.arange(16, dtype=np.float32).reshape(2, 8)
    assert np.array_equal(oracle.shared_ffn(z, z, np.zeros((8, 0), np.uint16), x, base), base)
    with pytest.raises(ValueError):
        oracle.shared_ffn(np.zeros((4, 8), np.uint16), np.zeros((4, 8), np.uint16), np.zeros((8, 5), np.uint16), x)
