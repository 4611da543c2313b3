"""Seeded synthetic workloads for the causal long convolution.

This module is shared by the test suite, the benchmark and the smoke check.
It draws random numbers and rounds them to the storage dtypes; it holds no
part of the convolution arithmetic, so neither the oracle nor the CUDA path
depends on the other through it.

Recipe (stated once here, restated in the design notes):

* Random source: the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014) used as a
  counter-based generator.  Element ``i`` of a stream is
  ``mix(base + (i + 1) * 0x9E3779B97F4A7C15)`` where ``base`` identifies the
  (seed, tensor) pair.  Every tensor has its own stream id, so tensors never
  share draws.
* Uniforms: ``((z >> 11) + 0.5) * 2**-53`` lies strictly inside (0, 1).
* Normals: Box-Muller on consecutive uniform pairs, in double precision.
* Rounding: values are produced in float64, rounded to float32
  (round-to-nearest-even), then to the tensor's 16-bit dtype
  (round-to-nearest-even).  Both the GPU path and the oracle see exactly these
  rounded values; the oracle widens them to double.

Workload shapes stand in for the FlashFFTConv page's benchmark inputs
(section 4: channel count 768 as in the Hyena / M2-BERT convolution
micro-benchmarks, the Path-512 sequence length 512*512, gene-length
sequences in the millions).  No dataset is read.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids of the tensors a workload draws (one stream per tensor).
STREAM_U = 1
STREAM_K = 2
STREAM_W_IN = 3
STREAM_W_OUT = 4
STREAM_ALPHA = 5
STREAM_SYMBOL = 6
STREAM_NOISE = 7

_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, stream: int) -> np.uint64:
    s = np.array([(int(seed) << 32) + int(stream)], dtype=np.uint64)
    return _mix(s * GOLDEN + np.uint64(0x632BE59BD9B4E019))[0]


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """``count`` raw 64-bit draws of stream ``stream`` starting at ``start``."""
    base = _stream_base(seed, stream)
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + idx * GOLDEN)


def uniform(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """Uniform doubles in (0, 1)."""
    out = np.empty(count, dtype=np.float64)
    for c0 in range(0, count, _CHUNK):
        c1 = min(count, c0 + _CHUNK)
        z = raw_u64(seed, stream, start + c0, c1 - c0)
        out[c0:c1] = ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    return out


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """Standard normal doubles by Box-Muller on uniform pairs."""
    out = np.empty(count, dtype=np.float64)
    npairs = (count + 1) // 2
    for p0 in range(0, npairs, _CHUNK // 2):
        p1 = min(npairs, p0 + _CHUNK // 2)
        u = uniform(seed, stream, 2 * (p1 - p0), start=2 * p0)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        th = (2.0 * math.pi) * u[1::2]
        pair = np.empty(2 * (p1 - p0), dtype=np.float64)
        pair[0::2] = r * np.cos(th)
        pair[1::2] = r * np.sin(th)
        lo, hi = 2 * p0, min(count, 2 * p1)
        out[lo:hi] = pair[: hi - lo]
    return out


# ---------------------------------------------------------------- rounding

def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        r = (b + bias) >> np.uint32(16)
    nan = np.isnan(x32)
    if nan.any():
        r = np.where(nan, np.uint32(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclasses.dataclass
class Rounded:
    """A tensor rounded to its storage dtype.

    ``bits`` holds the raw storage (uint16 for fp16/bf16, float32 for fp32);
    ``f64`` holds the same values widened exactly to double.
    """

    dtype: str
    bits: np.ndarray
    f64: np.ndarray


def round_to(x: np.ndarray, dtype: str) -> Rounded:
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "fp32":
        return Rounded(dtype, x32, x32.astype(np.float64))
    if dtype == "fp16":
        h = x32.astype(np.float16)
        return Rounded(dtype, h.view(np.uint16), h.astype(np.float64))
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x32)
        return Rounded(dtype, bits, bf16_bits_to_f64(bits))
    raise ValueError(f"unknown dtype {dtype!r}")


# ---------------------------------------------------------------- workloads

@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic causal-convolution workload.

    ``u_kind``: ``normal`` (u ~ N(0,1)) or ``onehot`` (4-symbol one-hot per
    group of 4 channels plus N(0, 0.1^2) noise).
    ``k_kind``: ``normal_scaled`` (k ~ N(0,1)/sqrt(N)) or ``decay``
    (k[h,t] = N(0,1) * exp(-alpha_h * t / N), alpha_h ~ U[1, 10]).
    """

    name: str
    B: int
    H: int
    N: int
    dtype: str
    gated: bool
    u_kind: str
    k_kind: str
    description: str

    @property
    def rows(self) -> int:
        return self.B * self.H

    @property
    def outputs(self) -> int:
        return self.B * self.H * self.N


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("causal-1k", 2, 8, 1024, "fp16", False, "normal", "normal_scaled",
                 "causal long conv, B=2 H=8 N=1024, fp16, no gating"),
        Workload("hyena-gated-4k", 8, 768, 4096, "bf16", True, "normal", "decay",
                 "Hyena-style gated conv y=w_out*conv(u*w_in,k), B=8 H=768 N=4096, bf16"),
        Workload("m2bert-16k", 16, 768, 16384, "fp16", False, "normal", "decay",
                 "M2-BERT-style conv, B=16 H=768 N=16384, fp16"),
        Workload("path512-256k", 4, 64, 262144, "bf16", False, "normal", "normal_scaled",
                 "Path-512-length conv (512x512 flattened), B=4 H=64 N=262144, bf16"),
        Workload("gene-2m", 1, 32, 2097152, "bf16", False, "onehot", "decay",
                 "gene-length conv, B=1 H=32 N=2097152, bf16 one-hot-like input"),
    ]
}

WORKLOAD_ORDER = ["causal-1k", "hyena-gated-4k", "m2bert-16k", "path512-256k", "gene-2m"]


def scaled(w: Workload, B: Optional[int] = None, H: Optional[int] = None,
           N: Optional[int] = None) -> Workload:
    """The same recipe at other sizes (for small parity cases)."""
    return dataclasses.replace(
        w, name=f"{w.name}[B={B or w.B},H={H or w.H},N={N or w.N}]",
        B=B or w.B, H=H or w.H, N=N or w.N)


def make_u(w: Workload, seed: int = 0) -> Rounded:
    n = w.B * w.H * w.N
    if w.u_kind == "normal":
        x = normal(seed, STREAM_U, n)
    elif w.u_kind == "onehot":
        if w.H % 4:
            raise ValueError("one-hot input needs H divisible by 4")
        groups = w.H // 4
        sym = np.floor(uniform(seed, STREAM_SYMBOL, w.B * groups * w.N) * 4.0).astype(np.int64)
        sym = np.minimum(sym, 3).reshape(w.B, groups, 1, w.N)
        onehot = (sym == np.arange(4).reshape(1, 1, 4, 1)).astype(np.float64)
        x = onehot.reshape(w.B, w.H, w.N).ravel() + 0.1 * normal(seed, STREAM_NOISE, n)
    else:
        raise ValueError(w.u_kind)
    return round_to(x.reshape(w.B, w.H, w.N), w.dtype)


def make_k(w: Workload, seed: int = 0) -> Rounded:
    g = normal(seed, STREAM_K, w.H * w.N).reshape(w.H, w.N)
    if w.k_kind == "normal_scaled":
        k = g / math.sqrt(w.N)
    elif w.k_kind == "decay":
        alpha = 1.0 + 9.0 * uniform(seed, STREAM_ALPHA, w.H)
        t = np.arange(w.N, dtype=np.float64) / w.N
        k = g * np.exp(-alpha[:, None] * t[None, :])
    else:
        raise ValueError(w.k_kind)
    return round_to(k, "fp32")


def make_gates(w: Workload, seed: int = 0):
    n = w.B * w.H * w.N
    w_in = round_to(normal(seed, STREAM_W_IN, n).reshape(w.B, w.H, w.N), w.dtype)
    w_out = round_to(normal(seed, STREAM_W_OUT, n).reshape(w.B, w.H, w.N), w.dtype)
    return w_in, w_out


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """All inputs of a workload: u, k and (if gated) w_in, w_out."""
    out = {"u": make_u(w, seed), "k": make_k(w, seed)}
    if w.gated:
        out["w_in"], out["w_out"] = make_gates(w, seed)
    return out
