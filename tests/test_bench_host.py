"""Host helpers of the benchmark (CPU, no GPU): the kernels one step
launches per path (the JSON line's gpu_launches), the algorithmic bytes of
the roofline, and the kept fraction of a frequency-sparse run's spectrum
against the oracle's band mask."""
import numpy as np
import pytest

import bench
import oracle
import workloads as W

F = pytest.importorskip("fft_long_convolution_gb300")


@pytest.mark.parametrize("N,order,launches", [
    (1024, 0, 1),        # fused, mma.sync
    (4096, 0, 1),        # fused, tcgen05
    (16384, 0, 1),
    (262144, 0, 3),      # passes A, B (tcgen05), C
    (262144, 4, 3),      # passes A, B (warp level), C
    (2097152, 0, 3),     # two-level outer factor, dense: fused A (RA and 64), B, fused C
])
def test_launches_per_step(N, order, launches):
    info = F.query(N, F.BF16, order)
    p = bench.path_of(info)
    assert p["launches_per_step"] == launches
    if info["path"] == F.PATH_MULTIPASS:
        # a sparse plan that skips every pair launches no pass B
        assert bench.path_of(info, 0)["launches_per_step"] == launches - 1
        assert bench.path_of(info, 3)["launches_per_step"] == launches


def test_launches_per_step_two_level_sparse():
    """A frequency-sparse two-level plan runs the same fused outer passes as
    the dense one (skipping dead sub-rows inside them): A, B, C, and no
    pass B when every pair is skipped."""
    info = F.query(2097152, F.BF16, 0)
    assert bench.path_of(info, 40, 256)["launches_per_step"] == 3
    assert "skipped" in bench.path_of(info, 40, 256)["kernel"]
    assert bench.path_of(info, 0, 256)["launches_per_step"] == 2
    assert bench.path_of(info, 256, 256)["launches_per_step"] == 3


def test_algorithmic_bytes():
    w = W.WORKLOADS["hyena-gated-4k"]
    a = bench.algorithmic(w)
    # u, w_in, w_out, y (2 bytes each) per row, plus the 16-bit spectrum once
    assert a["bytes"] == w.rows * w.N * 2 * 4 + w.H * (w.N + 1) * 4 == 213912576
    w = W.WORKLOADS["path512-256k"]
    assert bench.algorithmic(w)["bytes"] == w.rows * w.N * 2 * 2 + w.H * (w.N + 1) * 4


@pytest.mark.parametrize("name,band", [("path512-256k", [8, 33, 33]), ("gene-2m", [5, 8, 33, 33]),
                                       ("path512-256k", [3, 20, 7]), ("m2bert-16k", [20, 9, 9])])
def test_band_config_matches_the_mask(name, band):
    w = W.WORKLOADS[name]
    factors = F.query(w.N, F.F16 if w.dtype == "fp16" else F.BF16)["factors"]
    c = bench.config_of(w, band, factors)
    m = oracle.band_mask(w.N, factors, band)
    assert c["band"] == band
    assert c["spectrum_kept"] == pytest.approx(m[:w.N].mean(), rel=0, abs=1e-15)


def test_parse_band():
    assert bench.parse_band(None) is None
    assert bench.parse_band("") is None
    assert bench.parse_band("8,33,33") == [8, 33, 33]
