"""Pins of the oracle's partial convolution (CPU): brute-force windowed sums,
the limits T = 1 (scaling by k[0]) and T = N (the causal convolution), and a
shifted delta inside and beyond the window."""
import numpy as np
import pytest

import oracle


def _direct(u, k, T):
    N = u.size
    return np.array([sum(u[j] * k[t - j] for j in range(max(0, t - T + 1), t + 1)) for t in range(N)])


@pytest.mark.parametrize("N,T", [(8, 1), (8, 3), (64, 16), (256, 100), (256, 256)])
def test_partial_brute_force(N, T):
    rng = np.random.default_rng(N + T)
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    got = oracle.partial_conv(u, k, T)
    ref = _direct(u, k, T)
    assert np.allclose(got, ref, rtol=0, atol=1e-11)
    for t in (0, T - 1, N - 1):
        assert abs(oracle.direct_partial_conv_at(u, k, T, t) - ref[t]) < 1e-11


def test_partial_limits():
    rng = np.random.default_rng(5)
    N = 128
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    assert np.allclose(oracle.partial_conv(u, k, 1), k[0] * u, atol=1e-12)
    assert np.allclose(oracle.partial_conv(u, k, N), oracle.causal_conv(u, k), atol=1e-12)


@pytest.mark.parametrize("s,T", [(3, 8), (8, 8), (20, 8)])
def test_partial_shifted_delta(s, T):
    """k = delta_s: y[t] = u[t - s] if s < T (inside the window), else 0."""
    N = 64
    u = np.random.default_rng(s).standard_normal(N)
    k = np.zeros(N)
    k[s] = 1.0
    exp = np.zeros(N)
    if s < T:
        exp[s:] = u[: N - s]
    assert np.allclose(oracle.partial_conv(u, k, T), exp, atol=1e-12)
