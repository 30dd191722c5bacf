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
    # (1e8 + 1) + (-1e8) = 0 in float32 (1 is below half of 1e8's spacing)
    a = np.array([1e8, 1.0, -1e8], dtype=np.float32)
    assert stencil.window_sum_f32(a, 1, 3)[0] == np.float32(0.0)
    # (1 + 1e8) + (-1e8) = 0, whereas right to left, (-1e8 + 1e8) + 1, and
    # 1 + (1e8 + -1e8) both give 1: only the order as written gives 0
    b = np.array([1.0, 1e8, -1e8], dtype=np.float32)
    assert stencil.window_sum_f32(b, 1, 3)[0] == np.float32(0.0)


def test_planted_mistakes_are_caught(monkeypatch):
    """Each mistake, planted into the oracle itself, fails a pin above."""
    real = stencil.window_sum_f32

    def shifted(a, n_out, window=3):  # window starts one element late
        a = np.asarray(a, dtype=np.float32)
        return real(a[1:], n_out, window)

    def right_to_left(a, n_out, window=3):  # terms added in the reverse order
        a = np.asarray(a, dtype=np.float32)
        acc = a[window - 1:window - 1 + n_out].copy()
        for k in range(window - 2, -1, -1):
            acc = (acc + a[k:k + n_out]).astype(np.float32)
        return acc

    def short(a, n_out, window=3):  # one term dropped
        return real(a, n_out, max(1, window - 1))

    for mutant, pins in ((shifted, [test_page_shapes_and_definition]),
                         (right_to_left, [test_left_to_right_order_is_observable]),
                         (short, [test_page_shapes_and_definition,
                                  lambda: test_integer_inputs_match_exact_convolution(5)])):
        monkeypatch.setattr(stencil, "window_sum_f32", mutant)
        for pin in pins:
            with pytest.raises((AssertionError, ValueError)):
                pin()
        monkeypatch.setattr(stencil, "window_sum_f32", real)
    test_page_shapes_and_definition()  # the real oracle passes again
