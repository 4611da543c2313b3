"""Pins of the oracle's circular convolution (CPU): brute-force modular
sums, shifted deltas that wrap around, commutativity, and numpy's FFT as an
independent library."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("N", [1, 2, 8, 64])
def test_circular_brute_force(N):
    rng = np.random.default_rng(N)
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    ref = np.array([sum(u[j] * k[(t - j) % N] for j in range(N)) for t in range(N)])
    assert np.allclose(oracle.circular_conv(u, k), ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("s", [0, 1, 31, 63])
def test_circular_shifted_delta_wraps(s):
    N = 64
    u = np.random.default_rng(s).standard_normal(N)
    k = np.zeros(N)
    k[s] = 1.0
    assert np.allclose(oracle.circular_conv(u, k), np.roll(u, s), atol=1e-13)


def test_circular_commutes_and_matches_numpy():
    rng = np.random.default_rng(3)
    N = 1024
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    y = oracle.circular_conv(u, k)
    assert np.allclose(y, oracle.circular_conv(k, u), atol=1e-10)
    assert np.allclose(y, np.fft.ifft(np.fft.fft(u) * np.fft.fft(k)).real, atol=1e-10)
