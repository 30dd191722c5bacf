"""Pins of the window-sum oracle (no GPU).

MLC course "Ep7", section "Window Sum Example": B[i] = A[i] + A[i+1] + A[i+2],
A of 1027 float32, B of 1024.
"""
import numpy as np
import pytest

from oracle import stencil


def test_page_shapes_and_definition():
    a = np.arange(1027, dtype=np.float32)
    b = stencil.window_sum_f32(a, 1024, 3)
    assert b.shape == (1024,) and b.dtype == np.float32
    # closed form for A[i] = i: B[i] = 3 i + 3
    assert np.array_equal(b, 3 * np.arange(1024, dtype=np.float32) + 3)


@pytest.mark.parametrize("window", [1, 2, 3, 5, 17, 64])
def test_integer_inputs_match_exact_convolution(window):
    # small integers: every float32 partial sum is exact, so the result must
    # equal numpy's float64 convolution exactly
    rng = np.random.default_rng(window)
    n = 5000
    a = rng.integers(-1000, 1000, size=n + window - 1).astype(np.float32)
    want = np.convolve(a.astype(np.float64), np.ones(window), mode="valid")
    assert np.array_equal(stencil.window_sum_f32(a, n, window).astype(np.float64), want)


def test_random_floats_within_float32_rounding():
    rng = np.random.default_rng(3)
    n, window = 10000, 3
    a = rng.standard_normal(n + 2).astype(np.float32)
    got = stencil.window_sum_f32(a, n, window).astype(np.float64)
    exact = np.convolve(a.astype(np.float64), np.ones(window), mode="valid")
    # two float32 additions: error <= 2 u (|a|+|b|+|c|) with u = 2^-24
    bound = 2 * 2.0 ** -24 * np.convolve(np.abs(a.astype(np.float64)), np.ones(window), mode="valid")
    assert np.all(np.abs(got - exact) <= bound * (1 + 1e-12))


def test_left_to_right_order_is_observable():
    # (1e8 + 1) + (-1e8) = 0 in float32, while 1 + (1e8 + -1e8) would be 1
    a = np.array([1e8, 1.0, -1e8], dtype=np.float32)
    assert stencil.window_sum_f32(a, 1, 3)[0] == np.float32(0.0)


def test_planted_off_by_one_is_caught(monkeypatch):
    def shifted(a, n_out, window=3):
        a = np.asarray(a, dtype=np.float32)
        acc = a[1:n_out + 1].copy()
        for k in range(1, window):
            acc = (acc + a[k + 1:k + 1 + n_out]).astype(np.float32)
        return acc
    a = np.arange(1027 + 1, dtype=np.float32)
    assert not np.array_equal(shifted(a, 1024), 3 * np.arange(1024, dtype=np.float32) + 3)
