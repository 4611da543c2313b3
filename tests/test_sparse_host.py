"""Host logic of frequency-sparse plans (CPU, no GPU): which pairs of
sub-rows the multi-pass path still transforms, checked against a brute
force over the oracle's band mask, and argument validation."""
import numpy as np
import pytest

import oracle

F = pytest.importorskip("fft_long_convolution_gb300")


def _pairs_run_brute(N, factors, band):
    m = oracle.band_mask(N, factors, band)[:N]
    two_level = len(factors) == 4 and factors[3] == 64
    R0 = factors[0] * 64 if two_level else factors[0]
    live = m.reshape(N // R0, R0).any(axis=0)  # bin f = k0 + R0 q lives in sub-row k0
    run = 0
    for p in range(R0 // 2):
        partner = R0 - p if p else R0 // 2
        run += bool(live[p] or live[partner])
    return run, R0 // 2


CASES = [
    (65536, 0, [3, 33, 33]),
    (65536, 0, [4, 33, 33]),
    (262144, 0, [16, 33, 33]),
    (262144, 0, [9, 20, 7]),
    (262144, 0, [33, 33, 5]),
    (262144, 0, [1, 33, 33]),
    (262144, 0, [0, 33, 33]),
    (262144, 0, [20, 0, 33]),
    (524288, 0, [40, 33, 33]),
    (65536, 4, [2, 20, 9, 9]),
    (1048576, 0, [3, 16, 33, 33]),
    (1048576, 0, [1, 1, 33, 33]),
    (2097152, 0, [5, 16, 33, 33]),
    (2097152, 0, [2, 9, 33, 4]),
    (2097152, 0, [5, 33, 33, 33]),
]


@pytest.mark.parametrize("N,order,band", CASES)
def test_pairs_run_matches_brute_force(N, order, band):
    info = F.query(N, F.BF16, order)
    assert len(band) == info["order"]
    got = F.sparse_query(N, F.BF16, band, order)
    run, total = _pairs_run_brute(N, info["factors"], band)
    assert (got["pairs_run"], got["pairs_total"]) == (run, total)


def test_full_band_runs_every_pair():
    for N in (65536, 262144, 2097152):
        info = F.query(N, F.BF16)
        full = [Mj // 2 + 1 for Mj in info["factors"]]
        got = F.sparse_query(N, F.BF16, full)
        assert got["pairs_run"] == got["pairs_total"] > 0
        got = F.sparse_query(N, F.BF16, [b + 100 for b in full])  # clamped
        assert got["pairs_run"] == got["pairs_total"]


def test_fused_lengths_report_pairs_of_the_tensor_core_kernel():
    """The warp-level and 64 x 64 fused kernels report no pairs; the fused
    tensor-core kernel (N = 8192 .. 32768) reports R0 / 2 pairs of sub-rows
    (R0 = N / 4096) and, at R0 = 4, skips pair (1, 3) when the outer band
    keeps digit 0 alone."""
    for N in (1024, 4096):
        info = F.query(N, F.F16, order=3 if N < 4096 else 0)  # sparse patterns at 1K keep R1 x 16 x 16
        got = F.sparse_query(N, F.BF16, [1] * info["order"])
        assert got == {"pairs_run": 0, "pairs_total": 0}
    assert F.sparse_query(8192, F.BF16, [1, 1, 1]) == {"pairs_run": 1, "pairs_total": 1}
    assert F.sparse_query(16384, F.BF16, [1, 1, 1]) == {"pairs_run": 1, "pairs_total": 2}
    assert F.sparse_query(16384, F.BF16, [1, 33, 33]) == {"pairs_run": 1, "pairs_total": 2}
    assert F.sparse_query(16384, F.BF16, [2, 1, 1]) == {"pairs_run": 2, "pairs_total": 2}
    assert F.sparse_query(16384, F.BF16, [3, 0, 33]) == {"pairs_run": 1, "pairs_total": 2}  # inner axis empty
    assert F.sparse_query(32768, F.BF16, [1, 1, 1]) == {"pairs_run": 4, "pairs_total": 4}


@pytest.mark.parametrize("band", [[16, 33], [16, 33, 33, 33], [-1, 33, 33]])
def test_bad_band_is_invalid(band):
    with pytest.raises(F.FFTConvError) as e:
        F.sparse_query(262144, F.BF16, band)
    assert e.value.status == 1  # FFTCONV_ERR_INVALID
