"""Oracle for the causal long convolution (double precision, CPU).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm are the only callers.  The product
path never imports this package.

The arithmetic lives in ``fftconv_oracle.c`` (plain C, compiled here with the
system C compiler into ``oracle/_build/``).  This module only marshals numpy
arrays through ctypes; the C calls release the GIL, so rows can be spread
over threads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fftconv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library; returns its path."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        # -ffp-contract=off keeps every product and sum a separately rounded
        # double operation, exactly as written.
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64 = ctypes.c_int64
        lib.oracle_fft.argtypes = [_dp, _dp, i64, ctypes.c_int]
        lib.oracle_dft_direct.argtypes = [_dp, _dp, _dp, _dp, i64, ctypes.c_int]
        lib.oracle_causal_conv.argtypes = [_dp, _dp, _dp, i64]
        lib.oracle_causal_conv_gated.argtypes = [_dp, _dp, _dp, _dp, _dp, i64]
        lib.oracle_causal_conv_rows.argtypes = [_dp, _dp, _dp, _dp, _dp, i64, i64, i64, i64]
        lib.oracle_direct_causal_conv_at.argtypes = [_dp, _dp, i64, i64]
        lib.oracle_direct_causal_conv_at.restype = ctypes.c_double
        lib.oracle_direct_causal_conv.argtypes = [_dp, _dp, _dp, i64]
        lib.oracle_causal_corr.argtypes = [_dp, _dp, _dp, i64]
        lib.oracle_direct_causal_corr_at.argtypes = [_dp, _dp, i64, i64]
        lib.oracle_direct_causal_corr_at.restype = ctypes.c_double
        lib.oracle_input_grad_rows.argtypes = [_dp, _dp, _dp, _dp, _dp, i64, i64, i64, i64]
        lib.oracle_kernel_grad_channels.argtypes = [_dp, _dp, _dp, _dp, _dp, i64, i64, i64, i64, i64]
        lib.oracle_partial_conv.argtypes = [_dp, _dp, _dp, i64, i64]
        lib.oracle_direct_partial_conv_at.argtypes = [_dp, _dp, i64, i64, i64]
        lib.oracle_direct_partial_conv_at.restype = ctypes.c_double
        lib.oracle_circular_conv.argtypes = [_dp, _dp, _dp, i64]
        lib.oracle_masked_causal_conv.argtypes = [_dp, _dp, _dp, _dp, i64]
        lib.oracle_direct_masked_causal_conv.argtypes = [_dp, _dp, _dp, _dp, i64]
        lib.oracle_masked_causal_corr.argtypes = [_dp, _dp, _dp, _dp, i64]
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(_dp)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def fft(x: np.ndarray, inverse: bool = False) -> np.ndarray:
    """DFT (forward sign -1) or inverse DFT (sign +1, scaled 1/n), radix 2."""
    x = np.asarray(x, dtype=np.complex128)
    re, im = _f64(x.real).copy(), _f64(x.imag).copy()
    if _load().oracle_fft(_ptr(re), _ptr(im), re.size, 1 if inverse else -1):
        raise ValueError("length must be a power of two")
    return re + 1j * im


def dft_direct(x: np.ndarray, inverse: bool = False) -> np.ndarray:
    """Brute-force O(n^2) DFT, the definition written out."""
    x = np.asarray(x, dtype=np.complex128)
    re, im = _f64(x.real), _f64(x.imag)
    ore, oim = np.empty_like(re), np.empty_like(im)
    _load().oracle_dft_direct(_ptr(re), _ptr(im), _ptr(ore), _ptr(oim), re.size,
                              1 if inverse else -1)
    return ore + 1j * oim


def causal_conv(u: np.ndarray, k: np.ndarray) -> np.ndarray:
    """One row: y[t] = sum_{j<=t} u[j] k[t-j], through the 2N-point DFT."""
    u, k = _f64(u), _f64(k)
    y = np.empty_like(u)
    if _load().oracle_causal_conv(_ptr(u), _ptr(k), _ptr(y), u.size):
        raise ValueError("N must be a power of two")
    return y


def direct_causal_conv(u: np.ndarray, k: np.ndarray) -> np.ndarray:
    """One row by the O(N^2) definition."""
    u, k = _f64(u), _f64(k)
    y = np.empty_like(u)
    _load().oracle_direct_causal_conv(_ptr(u), _ptr(k), _ptr(y), u.size)
    return y


def direct_causal_conv_at(u: np.ndarray, k: np.ndarray, t: int) -> float:
    """One output y[t] by the definition (compensated sum), O(t)."""
    u, k = _f64(u), _f64(k)
    return float(_load().oracle_direct_causal_conv_at(_ptr(u), _ptr(k), u.size, int(t)))


def causal_conv_batch(u: np.ndarray, k: np.ndarray, w_in: Optional[np.ndarray] = None,
                      w_out: Optional[np.ndarray] = None, threads: int = 1,
                      rows: Optional[range] = None) -> np.ndarray:
    """u: [B, H, N] (or [rows, N] with H = k.shape[0]); k: [H, N].

    Returns y of u's shape (rows outside ``rows`` are left zero).  Gating is
    applied when both ``w_in`` and ``w_out`` are given.
    """
    k = _f64(k)
    H, N = k.shape
    u = _f64(u)
    shape = u.shape
    u2 = u.reshape(-1, N)
    gi = _f64(w_in).reshape(-1, N) if w_in is not None else None
    go = _f64(w_out).reshape(-1, N) if w_out is not None else None
    y = np.zeros_like(u2)
    nrows = u2.shape[0]
    todo = rows if rows is not None else range(nrows)
    lib = _load()

    def run(r0: int, r1: int):
        rc = lib.oracle_causal_conv_rows(_ptr(u2), _ptr(gi), _ptr(go), _ptr(k), _ptr(y),
                                         H, N, r0, r1)
        if rc:
            raise ValueError("oracle failed (N must be a power of two)")

    r_list = list(todo)
    if threads <= 1 or len(r_list) <= 1:
        for r in r_list:
            run(r, r + 1)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda r: run(r, r + 1), r_list))
    return y.reshape(shape)


# ---------------------------------------------------------------- backward

def causal_corr(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """One row: out[i] = sum_{t>=i} a[t] b[t-i], through the 2N-point DFT."""
    a, b = _f64(a), _f64(b)
    out = np.empty_like(a)
    if _load().oracle_causal_corr(_ptr(a), _ptr(b), _ptr(out), a.size):
        raise ValueError("N must be a power of two")
    return out


def direct_causal_corr_at(a: np.ndarray, b: np.ndarray, i: int) -> float:
    """One correlation output by the definition (compensated sum), O(N - i)."""
    a, b = _f64(a), _f64(b)
    return float(_load().oracle_direct_causal_corr_at(_ptr(a), _ptr(b), a.size, int(i)))


def input_grad_batch(dy: np.ndarray, k: np.ndarray, w_in: Optional[np.ndarray] = None,
                     w_out: Optional[np.ndarray] = None, threads: int = 1) -> np.ndarray:
    """du for dy [B, H, N], k [H, N]; gated when both gates are given:
    du = w_in * corr(w_out * dy, k)."""
    k = _f64(k)
    H, N = k.shape
    dy = _f64(dy)
    shape = dy.shape
    d2 = dy.reshape(-1, N)
    gi = _f64(w_in).reshape(-1, N) if w_in is not None else None
    go = _f64(w_out).reshape(-1, N) if w_out is not None else None
    du = np.zeros_like(d2)
    lib = _load()

    def run(r0: int, r1: int):
        rc = lib.oracle_input_grad_rows(_ptr(d2), _ptr(gi), _ptr(go), _ptr(k), _ptr(du), H, N, r0, r1)
        if rc:
            raise ValueError("oracle_input_grad_rows failed")

    _split(run, d2.shape[0], threads)
    return du.reshape(shape)


def kernel_grad(u: np.ndarray, dy: np.ndarray, w_in: Optional[np.ndarray] = None,
                w_out: Optional[np.ndarray] = None, threads: int = 1) -> np.ndarray:
    """dk [H, N] = sum_b corr(w_out * dy_b, w_in * u_b) for u, dy [B, H, N]."""
    u, dy = _f64(u), _f64(dy)
    B, H, N = u.shape
    gi = _f64(w_in) if w_in is not None else None
    go = _f64(w_out) if w_out is not None else None
    dk = np.zeros((H, N))
    lib = _load()

    def run(h0: int, h1: int):
        rc = lib.oracle_kernel_grad_channels(_ptr(u), _ptr(dy), _ptr(gi), _ptr(go), _ptr(dk), B, H, N, h0, h1)
        if rc:
            raise ValueError("oracle_kernel_grad_channels failed")

    _split(run, H, threads)
    return dk


def _split(run, n: int, threads: int):
    if threads <= 1 or n <= 1:
        run(0, n)
        return
    step = (n + threads - 1) // threads
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda r0: run(r0, min(n, r0 + step)), range(0, n, step)))


# ---------------------------------------------------------------- partial convolution

def partial_conv(u: np.ndarray, k: np.ndarray, T: int) -> np.ndarray:
    """One row: y[t] = sum_{t-T < j <= t} u[j] k[t-j] (k cut to T taps)."""
    u, k = _f64(u), _f64(k)
    y = np.empty_like(u)
    if _load().oracle_partial_conv(_ptr(u), _ptr(k), _ptr(y), u.size, int(T)):
        raise ValueError("N must be a power of two and 1 <= T <= N")
    return y


def direct_partial_conv_at(u: np.ndarray, k: np.ndarray, T: int, t: int) -> float:
    """One partial-convolution output by the definition, O(T)."""
    u, k = _f64(u), _f64(k)
    return float(_load().oracle_direct_partial_conv_at(_ptr(u), _ptr(k), u.size, int(T), int(t)))


# ---------------------------------------------------------------- circular convolution

def circular_conv(u: np.ndarray, k: np.ndarray) -> np.ndarray:
    """One row: y[t] = sum_j u[j] k[(t - j) mod N], through the N-point DFT."""
    u, k = _f64(u), _f64(k)
    y = np.empty_like(u)
    if _load().oracle_circular_conv(_ptr(u), _ptr(k), _ptr(y), u.size):
        raise ValueError("N must be a power of two")
    return y


# ---------------------------------------------------------------- frequency-sparse convolution

def band_mask(N: int, factors, band) -> np.ndarray:
    """Weights (0 or 1) of the spectrum bins f = 0..N for a frequency-sparse
    pattern on the decomposition's frequency digits (FlashFFTConv page,
    "Architectural Extensions", frequency-sparse part, and its pattern of
    zeroing whole rows along each axis of the reshaped k_f).

    The transform the decomposition runs has length M = N (complex, after
    the real-input packing); its frequency index r = f mod M is written in
    mixed radix over the factors, outer factor first:
    r = r_1 + M_1 r_2 + M_1 M_2 r_3 + ...  Bin f is kept when every digit is
    within its band in cyclic distance: min(r_j, M_j - r_j) < band[j].  A
    band of M_j/2 + 1 or more keeps the whole axis; a band of 0 zeroes it.
    """
    factors, band = [int(x) for x in factors], [int(x) for x in band]
    if len(factors) != len(band) or int(np.prod(factors)) != N:
        raise ValueError("one band per factor, and the factors must multiply to N")
    r = np.arange(N + 1, dtype=np.int64) % N
    keep = np.ones(N + 1, dtype=bool)
    for Mj, bj in zip(factors, band):
        d = r % Mj
        r = r // Mj
        keep &= np.minimum(d, Mj - d) < bj
    return keep.astype(np.float64)


def masked_causal_conv(u: np.ndarray, k: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """One row of the frequency-sparse convolution: the 2N-point spectrum of
    k weighted by mask[f] (f = 0..N, mirrored to 2N - f) before the product."""
    u, k, mask = _f64(u), _f64(k), _f64(mask)
    if mask.size != u.size + 1:
        raise ValueError("mask needs N + 1 entries")
    y = np.empty_like(u)
    if _load().oracle_masked_causal_conv(_ptr(u), _ptr(k), _ptr(mask), _ptr(y), u.size):
        raise ValueError("N must be a power of two")
    return y


def direct_masked_causal_conv(u: np.ndarray, k: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """The same row from DFT sums over bins 0..N (no FFT), O(N^2)."""
    u, k, mask = _f64(u), _f64(k), _f64(mask)
    if mask.size != u.size + 1:
        raise ValueError("mask needs N + 1 entries")
    y = np.empty_like(u)
    _load().oracle_direct_masked_causal_conv(_ptr(u), _ptr(k), _ptr(mask), _ptr(y), u.size)
    return y


def masked_causal_conv_batch(u: np.ndarray, k: np.ndarray, mask: np.ndarray, w_in: Optional[np.ndarray] = None,
                             w_out: Optional[np.ndarray] = None, threads: int = 1,
                             rows: Optional[range] = None) -> np.ndarray:
    """u: [B, H, N] (or [rows, N] with H = k.shape[0]), k: [H, N];
    y = w_out . masked_conv(u . w_in, k) per row (gates optional).  rows
    selects flat rows b*H + h (default all)."""
    u, k = _f64(u), _f64(k)
    H, N = k.shape
    R = u.size // N
    sel = list(rows) if rows is not None else list(range(R))
    uf = u.reshape(R, N)
    wi = _f64(w_in).reshape(R, N) if w_in is not None else None
    wo = _f64(w_out).reshape(R, N) if w_out is not None else None
    out = np.empty((len(sel), N))

    def run(i0, i1):
        for i in range(i0, i1):
            r = sel[i]
            x = uf[r] * wi[r] if wi is not None else uf[r]
            y = masked_causal_conv(x, k[r % H], mask)
            out[i] = y * wo[r] if wo is not None else y

    _split(run, len(sel), threads)
    return out


def masked_causal_corr(a: np.ndarray, b: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """One row of the masked causal correlation (the adjoint in u of the
    frequency-sparse convolution with kernel b)."""
    a, b, mask = _f64(a), _f64(b), _f64(mask)
    if mask.size != a.size + 1:
        raise ValueError("mask needs N + 1 entries")
    out = np.empty_like(a)
    if _load().oracle_masked_causal_corr(_ptr(a), _ptr(b), _ptr(mask), _ptr(out), a.size):
        raise ValueError("N must be a power of two")
    return out


def masked_input_grad_batch(dy: np.ndarray, k: np.ndarray, mask: np.ndarray, w_in: Optional[np.ndarray] = None,
                            w_out: Optional[np.ndarray] = None, threads: int = 1) -> np.ndarray:
    """Input gradient of y = w_out . masked_conv(u . w_in, k) for dy [B, H, N]:
    du = w_in . masked_corr(w_out . dy, k) per row (gates optional)."""
    dy, k = _f64(dy), _f64(k)
    B, H, N = dy.shape
    g = dy * _f64(w_out) if w_out is not None else dy
    gf = g.reshape(B * H, N)
    out = np.empty((B * H, N))

    def run(i0, i1):
        for r in range(i0, i1):
            out[r] = masked_causal_corr(gf[r], k[r % H], mask)

    _split(run, B * H, threads)
    out = out.reshape(B, H, N)
    return out * _f64(w_in) if w_in is not None else out
