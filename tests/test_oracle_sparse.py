"""Pins of the oracle's frequency-sparse convolution and of its band pattern
(CPU).  The masked convolution is pinned by hand-worked fixtures, by
single-bin closed forms (a cosine per kept bin, from direct sums), by a
brute-force DFT-sum route that uses no FFT, and by the all-ones mask reducing
to the plain convolution; the band pattern by hand-worked fixtures and by the
pages' sparsity formula."""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "freq_sparse.json")))


@pytest.mark.parametrize("case", GOLDEN["band_cases"], ids=lambda c: c["name"])
def test_band_golden(case):
    m = oracle.band_mask(case["N"], case["factors"], case["band"])
    assert m.shape == (case["N"] + 1,)
    assert list(np.nonzero(m)[0]) == case["kept"]
    assert set(np.unique(m)) <= {0.0, 1.0}


@pytest.mark.parametrize("case", GOLDEN["conv_cases"], ids=lambda c: c["name"])
def test_masked_conv_golden(case):
    y = oracle.masked_causal_conv(case["u"], case["k"], case["mask"])
    assert np.allclose(y, case["y"], rtol=0, atol=1e-14)
    yd = oracle.direct_masked_causal_conv(case["u"], case["k"], case["mask"])
    assert np.allclose(yd, case["y"], rtol=0, atol=1e-14)


def _kept_per_axis(Mj, bj):
    return sum(1 for d in range(Mj) if min(d, Mj - d) < bj)


@pytest.mark.parametrize("factors", [[4, 4], [64, 64], [16, 16, 16], [8, 64, 64], [4, 64, 64, 64]])
def test_band_count_matches_sparsity_formula(factors):
    # S = 1 - prod(kept_j) / prod(M_j): the pages' sparsity fraction of a
    # pattern that zeroes whole rows along each axis
    N = int(np.prod(factors))
    rng = np.random.default_rng(len(factors) * 1000 + factors[0])
    for _ in range(6):
        band = [int(rng.integers(0, Mj // 2 + 3)) for Mj in factors]
        m = oracle.band_mask(N, factors, band)
        kept = int(np.prod([_kept_per_axis(Mj, bj) for Mj, bj in zip(factors, band)]))
        assert int(m[:N].sum()) == kept
        assert m[N] == m[0]  # bin N has r = 0
        # closed form of the per-axis count
        for Mj, bj in zip(factors, band):
            assert _kept_per_axis(Mj, bj) == (0 if bj == 0 else min(Mj, 2 * bj - 1))


def test_band_full_keeps_everything():
    for factors in ([64, 64], [32, 16, 16], [8, 64, 64, 64]):
        N = int(np.prod(factors))
        assert oracle.band_mask(N, factors, [Mj // 2 + 1 for Mj in factors]).all()
        assert not oracle.band_mask(N, factors, [Mj // 2 for Mj in factors]).all()


def test_band_rejects_wrong_arguments():
    with pytest.raises(ValueError):
        oracle.band_mask(16, [4, 4], [1])
    with pytest.raises(ValueError):
        oracle.band_mask(32, [4, 4], [1, 1])


def _dft_bins(x):
    # U[f] = sum_n x[n] exp(-i pi f n / N), f = 0..N, by direct sums
    N = x.size
    f = np.arange(N + 1)[:, None]
    n = np.arange(N)[None, :]
    return (x[None, :] * np.exp(-1j * np.pi * ((f * n) % (2 * N)) / N)).sum(axis=1)


@pytest.mark.parametrize("N", [4, 16, 64])
def test_single_bin_closed_forms(N):
    rng = np.random.default_rng(N + 7)
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    U, K = _dft_bins(u), _dft_bins(k)
    t = np.arange(N)
    for f in (0, 1, N // 2, N - 1, N):
        mask = np.zeros(N + 1)
        mask[f] = 1.0
        if f in (0, N):
            ref = (U[f] * K[f]).real * np.cos(np.pi * f * t / N) / (2 * N)
        else:
            ref = (U[f] * K[f] * np.exp(1j * np.pi * f * t / N)).real / N
        for fn in (oracle.masked_causal_conv, oracle.direct_masked_causal_conv):
            got = fn(u, k, mask)
            assert np.allclose(got, ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max())), (fn.__name__, f)


@pytest.mark.parametrize("N", [8, 32, 128])
def test_fft_route_matches_dft_sums(N):
    rng = np.random.default_rng(N)
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    masks = [(rng.random(N + 1) < 0.5).astype(float), rng.standard_normal(N + 1), np.zeros(N + 1)]
    for m in masks:
        a = oracle.masked_causal_conv(u, k, m)
        b = oracle.direct_masked_causal_conv(u, k, m)
        assert np.allclose(a, b, rtol=0, atol=1e-12 * max(1.0, np.abs(b).max()))


@pytest.mark.parametrize("N", [1024, 4096])
def test_all_ones_is_the_plain_convolution(N):
    rng = np.random.default_rng(N)
    u, k = rng.standard_normal(N), rng.standard_normal(N) / np.sqrt(N)
    a = oracle.masked_causal_conv(u, k, np.ones(N + 1))
    b = oracle.causal_conv(u, k)
    assert np.allclose(a, b, rtol=0, atol=1e-12 * np.abs(b).max())
    for t in (0, 1, N // 3, N - 1):  # the definition, not a transform
        assert abs(a[t] - oracle.direct_causal_conv_at(u, k, t)) <= 1e-11 * max(1.0, np.abs(b).max())


def test_band_mask_is_a_projection():
    # masking twice changes nothing; complementary masks add up to the plain result
    N, factors = 256, [4, 8, 8]
    rng = np.random.default_rng(5)
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    m = oracle.band_mask(N, factors, [1, 3, 2])
    full = oracle.causal_conv(u, k)
    ya = oracle.masked_causal_conv(u, k, m)
    yb = oracle.masked_causal_conv(u, k, 1.0 - m)
    assert np.allclose(ya + yb, full, rtol=0, atol=1e-12 * np.abs(full).max())
    assert 0 < m.sum() < N + 1


def test_batch_rows_use_their_channel_and_gates():
    B, H, N = 2, 3, 64
    rng = np.random.default_rng(1)
    u, wi, wo = (rng.standard_normal((B, H, N)) for _ in range(3))
    k = rng.standard_normal((H, N))
    m = oracle.band_mask(N, [8, 8], [2, 3])
    y = oracle.masked_causal_conv_batch(u, k, m, wi, wo, threads=2)
    for r in range(B * H):
        b, h = divmod(r, H)
        ref = wo[b, h] * oracle.direct_masked_causal_conv(u[b, h] * wi[b, h], k[h], m)
        assert np.allclose(y[r], ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))


SPARSE_MUTANTS = {
    "mask not mirrored to the upper half": ("double w = f <= N ? mask[f] : mask[L2 - f];",
                                            "double w = f <= N ? mask[f] : 1.0;"),
    "mirror off by one": ("double w = f <= N ? mask[f] : mask[L2 - f];",
                          "double w = f <= N ? mask[f] : mask[L2 - f - 1];"),
    "mask on the real part only": ("double pi = (ur[f] * ki[f] + ui[f] * kr[f]) * w;",
                                   "double pi = (ur[f] * ki[f] + ui[f] * kr[f]);"),
    "direct sums: conjugated U": ("Ur += u[n] * c; Ui -= u[n] * s;", "Ur += u[n] * c; Ui += u[n] * s;"),
    "direct sums: mirror weight dropped": ("s += 2.0 * (pr[f] * cos(a) - pi[f] * sin(a));",
                                           "s += (pr[f] * cos(a) - pi[f] * sin(a));"),
    "direct sums: Nyquist sign": ("double s = pr[0] + ((t & 1) ? -pr[N] : pr[N]);",
                                  "double s = pr[0] + pr[N];"),
}


def _sparse_pins_pass(lib) -> bool:
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    ok = True
    for case in GOLDEN["conv_cases"]:
        u, k, m = (np.array(case[x], dtype=float) for x in ("u", "k", "mask"))
        for fn in (lib.oracle_masked_causal_conv, lib.oracle_direct_masked_causal_conv):
            y = np.zeros(u.size)
            fn(P(u), P(k), P(m), P(y), ctypes.c_int64(u.size))
            ok &= bool(np.allclose(y, case["y"], rtol=0, atol=1e-12))
    N = 16
    rng = np.random.default_rng(3)
    u, k = rng.standard_normal(N), rng.standard_normal(N)
    U, K = _dft_bins(u), _dft_bins(k)
    t = np.arange(N)
    for f in (0, 3, N):
        m = np.zeros(N + 1)
        m[f] = 1.0
        ref = ((U[f] * K[f] * np.exp(1j * np.pi * f * t / N)).real / N) * (0.5 if f in (0, N) else 1.0)
        for fn in (lib.oracle_masked_causal_conv, lib.oracle_direct_masked_causal_conv):
            y = np.zeros(N)
            fn(P(u), P(k), P(m), P(y), ctypes.c_int64(N))
            ok &= bool(np.allclose(y, ref, rtol=0, atol=1e-12))
    return ok


def test_pins_catch_planted_mistakes(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fftconv_oracle.c")).read()
    base = tmp_path / "base.c"
    base.write_text(src)
    subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", str(base), "-o", str(base) + ".so", "-lm"])
    assert _sparse_pins_pass(ctypes.CDLL(str(base) + ".so"))
    for name, (old, new) in SPARSE_MUTANTS.items():
        assert src.count(old) == 1, name
        path = tmp_path / f"m_{abs(hash(name))}.c"
        path.write_text(src.replace(old, new))
        subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", str(path), "-o", str(path) + ".so", "-lm"])
        assert not _sparse_pins_pass(ctypes.CDLL(str(path) + ".so")), f"planted mistake not caught: {name}"


BAND_MUTANTS = {
    "axes taken inner first": ("for Mj, bj in zip(factors, band):", "for Mj, bj in zip(factors[::-1], band[::-1]):"),
    "band edge included": ("keep &= np.minimum(d, Mj - d) < bj", "keep &= np.minimum(d, Mj - d) <= bj"),
    "distance not cyclic": ("keep &= np.minimum(d, Mj - d) < bj", "keep &= d < bj"),
    "cut applied after the next axis's digit": ("d = r % Mj\n        r = r // Mj", "r = r // Mj\n        d = r % Mj"),
}


def test_band_pins_catch_planted_mistakes():
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle.band_mask))

    def fixtures_pass(fn):
        for case in GOLDEN["band_cases"]:
            try:
                m = fn(case["N"], case["factors"], case["band"])
            except Exception:
                return False
            if list(np.nonzero(m)[0]) != case["kept"]:
                return False
        return True

    assert fixtures_pass(oracle.band_mask)
    for name, (old, new) in BAND_MUTANTS.items():
        assert src.count(old) == 1, name
        ns = {"np": np}
        exec(src.replace(old, new), ns)
        assert not fixtures_pass(ns["band_mask"]), f"planted mistake not caught: {name}"


# ---------------------------------------------------------------- adjoint (input gradient)

@pytest.mark.parametrize("N,factors,band", [(64, [8, 8], [2, 3]), (256, [4, 8, 8], [1, 3, 2]), (1024, [32, 32], [9, 17])])
def test_masked_corr_is_the_adjoint(N, factors, band):
    # <dy, A_m u> = <A_m^T dy, u>, with A_m the masked convolution (pinned above)
    rng = np.random.default_rng(N)
    m = oracle.band_mask(N, factors, band)
    for _ in range(3):
        u, dy, k = rng.standard_normal(N), rng.standard_normal(N), rng.standard_normal(N)
        lhs = float(dy @ oracle.masked_causal_conv(u, k, m))
        rhs = float(u @ oracle.masked_causal_corr(dy, k, m))
        assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs), float(np.abs(dy).sum() * np.abs(u).sum()) * 1e-3)


def test_masked_corr_all_ones_is_the_correlation():
    rng = np.random.default_rng(2)
    N = 512
    a, b = rng.standard_normal(N), rng.standard_normal(N)
    got = oracle.masked_causal_corr(a, b, np.ones(N + 1))
    ref = oracle.causal_corr(a, b)
    assert np.allclose(got, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    for i in (0, 1, N // 2, N - 1):  # the definition, not a transform
        assert abs(got[i] - oracle.direct_causal_corr_at(a, b, i)) <= 1e-11 * np.abs(ref).max()


def test_masked_input_grad_gates():
    B, H, N = 2, 3, 64
    rng = np.random.default_rng(4)
    dy, wi, wo = (rng.standard_normal((B, H, N)) for _ in range(3))
    k = rng.standard_normal((H, N))
    m = oracle.band_mask(N, [8, 8], [3, 2])
    du = oracle.masked_input_grad_batch(dy, k, m, wi, wo, threads=2)
    for b in range(B):
        for h in range(H):
            ref = wi[b, h] * oracle.masked_causal_corr(wo[b, h] * dy[b, h], k[h], m)
            assert np.allclose(du[b, h], ref, rtol=0, atol=1e-12 * max(1.0, np.abs(ref).max()))


CORR_MUTANTS = {
    "correlation weight not mirrored": ("double wgt = f <= N ? mask[f] : mask[L2 - f];",
                                        "double wgt = f <= N ? mask[f] : 1.0;"),
    "correlation without the conjugate": ("double ci = (ai[f] * br[f] - ar[f] * bi[f]) * wgt;",
                                          "double ci = (ai[f] * br[f] + ar[f] * bi[f]) * wgt;"),
    "weight on the real part only": ("double ci = (ai[f] * br[f] - ar[f] * bi[f]) * wgt;",
                                     "double ci = (ai[f] * br[f] - ar[f] * bi[f]);"),
}


def _corr_pins_pass(lib) -> bool:
    P = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    rng = np.random.default_rng(8)
    N = 64
    m = oracle.band_mask(N, [8, 8], [2, 3])
    ok = True
    for _ in range(2):
        u, dy, k = rng.standard_normal(N), rng.standard_normal(N), rng.standard_normal(N)
        y, du = np.zeros(N), np.zeros(N)
        lib.oracle_masked_causal_conv(P(u), P(k), P(m), P(y), ctypes.c_int64(N))
        lib.oracle_masked_causal_corr(P(dy), P(k), P(m), P(du), ctypes.c_int64(N))
        ok &= abs(float(dy @ y) - float(u @ du)) <= 1e-10 * max(1.0, abs(float(dy @ y)))
    return bool(ok)


def test_corr_pins_catch_planted_mistakes(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fftconv_oracle.c")).read()
    base = tmp_path / "base.c"
    base.write_text(src)
    subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", str(base), "-o", str(base) + ".so", "-lm"])
    assert _corr_pins_pass(ctypes.CDLL(str(base) + ".so"))
    for name, (old, new) in CORR_MUTANTS.items():
        assert src.count(old) == 1, name
        path = tmp_path / f"m_{abs(hash(name))}.c"
        path.write_text(src.replace(old, new))
        subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", str(path), "-o", str(path) + ".so", "-lm"])
        assert not _corr_pins_pass(ctypes.CDLL(str(path) + ".so")), f"planted mistake not caught: {name}"
