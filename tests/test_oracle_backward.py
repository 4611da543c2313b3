"""Pins of the oracle's backward pass (CPU).  The gradients are pinned by
the identities that define them (the adjoint of the convolution in u and in
k), by brute-force sums on small sizes and by shifted-delta kernels; none of
these retypes the oracle's DFT route."""
import numpy as np
import pytest

import oracle


def _direct_corr(a, b):
    N = a.size
    return np.array([sum(a[t] * b[t - i] for t in range(i, N)) for i in range(N)])


def _direct_conv(u, k):
    N = u.size
    return np.array([sum(u[j] * k[t - j] for j in range(t + 1)) for t in range(N)])


@pytest.mark.parametrize("N", [1, 2, 8, 64, 256])
def test_corr_brute_force(N):
    rng = np.random.default_rng(N)
    a, b = rng.standard_normal(N), rng.standard_normal(N)
    got = oracle.causal_corr(a, b)
    ref = _direct_corr(a, b)
    assert np.allclose(got, ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))
    for i in (0, N // 2, N - 1):
        assert abs(oracle.direct_causal_corr_at(a, b, i) - ref[i]) <= 1e-12 * max(1.0, abs(ref[i]))


@pytest.mark.parametrize("N", [64, 1024])
def test_input_grad_is_the_adjoint_of_the_convolution(N):
    """<conv(u, k), dy> = <u, du> for every u: du is the gradient in u."""
    rng = np.random.default_rng(7)
    u, k, dy = rng.standard_normal(N), rng.standard_normal(N), rng.standard_normal(N)
    du = oracle.input_grad_batch(dy[None, None], k[None])[0, 0]
    lhs = float(np.dot(oracle.causal_conv(u, k), dy))
    assert abs(lhs - float(np.dot(u, du))) <= 1e-10 * (abs(lhs) + np.abs(u).sum())


def test_gated_gradients_are_adjoints():
    """y = w_out * conv(u * w_in, k): the derivative of sum(dy * y) along
    any du (any dk) equals <du_oracle, du> (<dk_oracle, dk>)."""
    rng = np.random.default_rng(8)
    B, H, N = 3, 2, 128
    u, dy = rng.standard_normal((B, H, N)), rng.standard_normal((B, H, N))
    wi, wo = rng.standard_normal((B, H, N)), rng.standard_normal((B, H, N))
    k = rng.standard_normal((H, N))

    def loss(u_, k_):
        return float((dy * oracle.causal_conv_batch(u_, k_, wi, wo)).sum())

    du = oracle.input_grad_batch(dy, k, wi, wo)
    dk = oracle.kernel_grad(u, dy, wi, wo)
    v = rng.standard_normal((B, H, N))
    assert abs(loss(v, k) - float((du * v).sum())) <= 1e-9 * np.abs(du * v).sum()  # loss is linear in u
    kv = rng.standard_normal((H, N))
    assert abs(loss(u, kv) - float((dk * kv).sum())) <= 1e-9 * np.abs(dk * kv).sum()  # and in k


def test_kernel_grad_brute_force_sum_over_batch():
    rng = np.random.default_rng(9)
    B, H, N = 4, 3, 32
    u, dy = rng.standard_normal((B, H, N)), rng.standard_normal((B, H, N))
    dk = oracle.kernel_grad(u, dy, threads=2)
    for h in range(H):
        ref = sum(_direct_corr(dy[b, h], u[b, h]) for b in range(B))
        assert np.allclose(dk[h], ref, rtol=0, atol=1e-11)


@pytest.mark.parametrize("s", [0, 1, 17, 63])
def test_input_grad_shifted_delta(s):
    """k = delta_s: du[j] = dy[j + s] for j + s < N, 0 above (causality)."""
    N = 64
    dy = np.random.default_rng(s).standard_normal(N)
    k = np.zeros(N)
    k[s] = 1.0
    du = oracle.input_grad_batch(dy[None, None], k[None])[0, 0]
    exp = np.zeros(N)
    exp[: N - s] = dy[s:]
    assert np.allclose(du, exp, rtol=0, atol=1e-13)


def test_direct_conv_and_corr_are_mutual_adjoints_brute_force():
    rng = np.random.default_rng(10)
    N = 16
    u, k, dy = rng.standard_normal(N), rng.standard_normal(N), rng.standard_normal(N)
    assert abs(np.dot(_direct_conv(u, k), dy) - np.dot(u, _direct_corr(dy, k))) < 1e-12


BACKWARD_MUTANTS = {
    "correlation without the conjugate": ("double pi = ai[i] * br[i] - ar[i] * bi[i];",
                                          "double pi = ai[i] * br[i] + ar[i] * bi[i];"),
    "correlation without zero padding": ("const int64_t L2 = 2 * N;", "const int64_t L2 = N;"),
    "input gradient gate swapped": ("g[t] = w_out ? dy[r * N + t] * w_out[r * N + t] : dy[r * N + t];\n        int rc",
                                    "g[t] = w_out ? dy[r * N + t] * w_in[r * N + t] : dy[r * N + t];\n        int rc"),
    "kernel gradient misses a batch row": ("for (int64_t b = 0; b < B; ++b) {", "for (int64_t b = 1; b < B; ++b) {"),
    "direct sum starts one late": ("for (int64_t t = i; t < N; ++t) {", "for (int64_t t = i + 1; t < N; ++t) {"),
}


def _backward_pins_pass(lib) -> bool:
    import ctypes
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    lib.oracle_direct_causal_corr_at.restype = ctypes.c_double
    rng = np.random.default_rng(0)
    ok = True
    B, H, N = 3, 2, 32
    u, dy = rng.standard_normal((B, H, N)), rng.standard_normal((B, H, N))
    wi, wo = rng.standard_normal((B, H, N)), rng.standard_normal((B, H, N))
    k = rng.standard_normal((H, N))
    for gated in (False, True):
        gi, go = (wi, wo) if gated else (None, None)
        du = np.zeros((B * H, N))
        lib.oracle_input_grad_rows(P(dy), P(gi) if gated else None, P(go) if gated else None, P(k), P(du),
                                   ctypes.c_int64(H), ctypes.c_int64(N), ctypes.c_int64(0), ctypes.c_int64(B * H))
        dk = np.zeros((H, N))
        lib.oracle_kernel_grad_channels(P(u), P(dy), P(gi) if gated else None, P(go) if gated else None, P(dk),
                                        ctypes.c_int64(B), ctypes.c_int64(H), ctypes.c_int64(N), ctypes.c_int64(0),
                                        ctypes.c_int64(H))
        g = dy * wo if gated else dy
        x = u * wi if gated else u
        for b in range(B):
            for h in range(H):
                ref = _direct_corr(g[b, h], k[h]) * (wi[b, h] if gated else 1.0)
                ok &= np.allclose(du[b * H + h], ref, atol=1e-10)
        for h in range(H):
            ref = sum(_direct_corr(g[b, h], x[b, h]) for b in range(B))
            ok &= np.allclose(dk[h], ref, atol=1e-10)
    a, c = rng.standard_normal(N), rng.standard_normal(N)
    ref = _direct_corr(a, c)
    for i in range(N):
        ok &= abs(lib.oracle_direct_causal_corr_at(P(a), P(c), ctypes.c_int64(N), ctypes.c_int64(i)) - ref[i]) < 1e-10
    return bool(ok)


def test_backward_pins_catch_planted_mistakes(tmp_path):
    import ctypes
    import os
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fftconv_oracle.c")).read()
    base = tmp_path / "base.c"
    base.write_text(src)
    subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", str(base), "-o", str(base) + ".so", "-lm"])
    assert _backward_pins_pass(ctypes.CDLL(str(base) + ".so"))
    for name, (old, new) in BACKWARD_MUTANTS.items():
        assert src.count(old) == 1, name
        path = tmp_path / f"m_{abs(hash(name))}.c"
        path.write_text(src.replace(old, new))
        subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", str(path), "-o", str(path) + ".so", "-lm"])
        assert not _backward_pins_pass(ctypes.CDLL(str(path) + ".so")), f"planted mistake not caught: {name}"
