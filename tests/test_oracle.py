"""Pins for the oracle (CPU only).

Each check ties the oracle to something other than itself: brute force on
tiny inputs, numpy's FFT (an independent library), closed forms, invariants
and hand-worked fixtures (tests/golden/).  The last test plants mistakes in a
copy of the oracle's C source and checks that the pins catch every one.
"""
import ctypes
import json
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "causal_conv_small.json")
rng = np.random.default_rng(1234)


def _rel(a, b):
    return np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(np.asarray(b)), 1e-300)


# ------------------------------------------------------------ DFT pins

@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 64, 256, 1024])
def test_fft_matches_bruteforce_dft(n):
    x = rng.standard_normal(n) + 1j * rng.standard_normal(n)
    assert _rel(oracle.fft(x), oracle.dft_direct(x)) < 1e-12
    assert _rel(oracle.fft(x, inverse=True), oracle.dft_direct(x, inverse=True)) < 1e-12


@pytest.mark.parametrize("n", [2, 32, 4096, 1 << 16])
def test_fft_matches_numpy(n):
    x = rng.standard_normal(n) + 1j * rng.standard_normal(n)
    assert _rel(oracle.fft(x), np.fft.fft(x)) < 1e-12
    assert _rel(oracle.fft(x, inverse=True), np.fft.ifft(x)) < 1e-12


def test_bruteforce_dft_matches_numpy_odd_length():
    x = rng.standard_normal(15) + 1j * rng.standard_normal(15)
    assert _rel(oracle.dft_direct(x), np.fft.fft(x)) < 1e-12


def test_dft_golden():
    for c in json.load(open(GOLDEN))["dft_cases"]:
        x = np.array(c["x_re"]) + 1j * np.array(c["x_im"])
        X = np.array(c["X_re"]) + 1j * np.array(c["X_im"])
        np.testing.assert_allclose(oracle.fft(x), X, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(oracle.dft_direct(x), X, atol=1e-12, err_msg=c["name"])


@pytest.mark.parametrize("n", [16, 1024])
def test_single_tone(n):
    for f in [0, 1, n // 3, n - 1]:
        x = np.exp(2j * np.pi * f * np.arange(n) / n)
        expect = np.zeros(n, complex)
        expect[f] = n
        np.testing.assert_allclose(oracle.fft(x), expect, atol=1e-9)


def test_inverse_roundtrip_and_parseval():
    n = 1 << 14
    x = rng.standard_normal(n) + 1j * rng.standard_normal(n)
    X = oracle.fft(x)
    assert _rel(oracle.fft(X, inverse=True), x) < 1e-13
    assert abs(np.sum(np.abs(x) ** 2) - np.sum(np.abs(X) ** 2) / n) / np.sum(np.abs(x) ** 2) < 1e-13


def test_fft_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        oracle.fft(np.ones(12))


# ------------------------------------------------------------ convolution pins

def test_conv_golden():
    for c in json.load(open(GOLDEN))["cases"]:
        u = np.array(c["u"], float)
        k = np.array(c["k"], float)
        if "w_in" in c:
            y = oracle.causal_conv_batch(u[None, None], k[None], np.array(c["w_in"])[None, None],
                                         np.array(c["w_out"])[None, None])[0, 0]
        else:
            y = oracle.causal_conv(u, k)
            np.testing.assert_allclose(oracle.direct_causal_conv(u, k), c["y"], atol=1e-14)
        np.testing.assert_allclose(y, c["y"], atol=1e-12, err_msg=c["name"])


@pytest.mark.parametrize("logn", range(0, 13))
def test_conv_matches_direct(logn):
    N = 1 << logn
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    y = oracle.causal_conv(u, k)
    yd = oracle.direct_causal_conv(u, k)
    assert np.max(np.abs(y - yd)) <= 1e-12 * max(1.0, np.max(np.abs(yd))) * max(1, logn)


def test_conv_matches_numpy_fft_pipeline():
    """Independent pipeline: numpy's real FFT of size 2N (library routine)."""
    N = 1 << 13
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    ref = np.fft.irfft(np.fft.rfft(u, 2 * N) * np.fft.rfft(k, 2 * N), 2 * N)[:N]
    assert _rel(oracle.causal_conv(u, k), ref) < 1e-12


@pytest.mark.parametrize("N", [16, 1024, 1 << 15])
def test_delta_and_shifted_delta(N):
    u = rng.standard_normal(N)
    for s in [0, 1, N // 2, N - 1]:
        k = np.zeros(N)
        k[s] = 1.0
        expect = np.zeros(N)
        expect[s:] = u[: N - s]
        np.testing.assert_allclose(oracle.causal_conv(u, k), expect, atol=1e-12)


def test_u_delta_returns_kernel():
    N = 4096
    k = rng.standard_normal(N)
    u = np.zeros(N)
    u[0] = 1.0
    np.testing.assert_allclose(oracle.causal_conv(u, k), k, atol=1e-12)


def test_constant_input_prefix_sum():
    N = 2048
    k = rng.standard_normal(N)
    np.testing.assert_allclose(oracle.causal_conv(np.ones(N), k), np.cumsum(k), atol=1e-10)


def test_linearity_and_commutativity():
    N = 1 << 12
    u1, u2, k1, k2 = (rng.standard_normal(N) for _ in range(4))
    a, b = 0.75, -2.5
    lhs = oracle.causal_conv(a * u1 + b * u2, k1)
    rhs = a * oracle.causal_conv(u1, k1) + b * oracle.causal_conv(u2, k1)
    assert _rel(lhs, rhs) < 1e-12
    lhs = oracle.causal_conv(u1, a * k1 + b * k2)
    rhs = a * oracle.causal_conv(u1, k1) + b * oracle.causal_conv(u1, k2)
    assert _rel(lhs, rhs) < 1e-12
    assert _rel(oracle.causal_conv(u1, k1), oracle.causal_conv(k1, u1)) < 1e-12


def test_causality():
    """Changing u after position t leaves y[0..t] unchanged."""
    N = 1024
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    u2 = u.copy()
    u2[600:] = rng.standard_normal(N - 600)
    y, y2 = oracle.causal_conv(u, k), oracle.causal_conv(u2, k)
    np.testing.assert_allclose(y[:600], y2[:600], atol=1e-12)
    assert np.max(np.abs(y[600:] - y2[600:])) > 1e-3


def test_direct_at_large_n_sampled():
    """At N = 2^18 the FFT oracle agrees with the definition at sampled t."""
    N = 1 << 18
    u, k = rng.standard_normal(N), rng.standard_normal(N) / np.sqrt(N)
    y = oracle.causal_conv(u, k)
    for t in [0, 1, 777, N // 2, N - 2, N - 1] + list(rng.integers(0, N, 20)):
        ref = oracle.direct_causal_conv_at(u, k, int(t))
        assert abs(y[t] - ref) <= 1e-11 * max(1.0, abs(ref))


def test_batch_rows_use_their_channel():
    B, H, N = 2, 3, 64
    u = rng.standard_normal((B, H, N))
    k = rng.standard_normal((H, N))
    wi, wo = rng.standard_normal((B, H, N)), rng.standard_normal((B, H, N))
    y = oracle.causal_conv_batch(u, k, threads=2)
    yg = oracle.causal_conv_batch(u, k, wi, wo)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(y[b, h], oracle.direct_causal_conv(u[b, h], k[h]), atol=1e-12)
            np.testing.assert_allclose(
                yg[b, h], wo[b, h] * oracle.direct_causal_conv(u[b, h] * wi[b, h], k[h]), atol=1e-12)


# ------------------------------------------------------------ planted mistakes

MUTANTS = {
    "twiddle sign flipped": ("double ang = sign * 2.0 * ORACLE_PI * (double)j / (double)len;",
                             "double ang = -sign * 2.0 * ORACLE_PI * (double)j / (double)len;"),
    "butterfly difference dropped": ("re[b] = re[a] - tr;", "re[b] = re[a] + tr;"),
    "inverse scale dropped": ("re[i] /= (double)n; im[i] /= (double)n;", "(void)0;"),
    "no zero padding (circular)": ("int64_t L = 2 * N;", "int64_t L = N;"),
    "pointwise product transposed imag": ("double pi = ur[i] * ki[i] + ui[i] * kr[i];",
                                          "double pi = ur[i] * ki[i] - ui[i] * kr[i];"),
    "bit reversal skipped": ("if (i < j) {", "if (0) {"),
    "off-by-one in direct sum": ("for (int64_t j = 0; j <= t; ++j)", "for (int64_t j = 0; j < t; ++j)"),
    "gate applied to wrong tensor": ("x[i] = u[i] * w_in[i];", "x[i] = u[i] * w_out[i];"),
}


def _pins_pass(lib) -> bool:
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_causal_conv.argtypes = [dp, dp, dp, ctypes.c_int64]
    lib.oracle_fft.argtypes = [dp, dp, ctypes.c_int64, ctypes.c_int]
    lib.oracle_direct_causal_conv_at.argtypes = [dp, dp, ctypes.c_int64, ctypes.c_int64]
    lib.oracle_direct_causal_conv_at.restype = ctypes.c_double
    lib.oracle_causal_conv_gated.argtypes = [dp, dp, dp, dp, dp, ctypes.c_int64]

    def P(a):
        return a.ctypes.data_as(dp)

    ok = True
    golden = json.load(open(GOLDEN))
    for c in golden["dft_cases"]:
        re = np.array(c["x_re"], float)
        im = np.array(c["x_im"], float)
        lib.oracle_fft(P(re), P(im), re.size, -1)
        ok &= np.allclose(re, c["X_re"], atol=1e-9) and np.allclose(im, c["X_im"], atol=1e-9)
    x = rng.standard_normal(64) + 1j * rng.standard_normal(64)
    re, im = x.real.copy(), x.imag.copy()
    lib.oracle_fft(P(re), P(im), 64, 1)
    ok &= np.allclose(re + 1j * im, np.fft.ifft(x), atol=1e-9)
    for c in golden["cases"]:
        u = np.array(c["u"], float)
        k = np.array(c["k"], float)
        y = np.empty_like(u)
        if "w_in" in c:
            wi, wo = np.array(c["w_in"], float), np.array(c["w_out"], float)
            lib.oracle_causal_conv_gated(P(u), P(wi), P(wo), P(k), P(y), u.size)
        else:
            lib.oracle_causal_conv(P(u), P(k), P(y), u.size)
            for t in range(u.size):
                ok &= abs(lib.oracle_direct_causal_conv_at(P(u), P(k), u.size, t) - c["y"][t]) < 1e-9
        ok &= np.allclose(y, c["y"], atol=1e-9)
    return bool(ok)


def test_pins_catch_planted_mistakes(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fftconv_oracle.c")).read()
    # the unmodified source passes the same checks
    base = tmp_path / "base.so"
    (tmp_path / "base.c").write_text(src)
    subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", str(tmp_path / "base.c"), "-o", str(base), "-lm"])
    assert _pins_pass(ctypes.CDLL(str(base)))
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, name
        path = tmp_path / f"m_{abs(hash(name))}.c"
        path.write_text(src.replace(old, new))
        so = str(path) + ".so"
        subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", str(path), "-o", so, "-lm"])
        assert not _pins_pass(ctypes.CDLL(so)), f"planted mistake not caught: {name}"
