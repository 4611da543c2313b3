"""The C-ABI library: loads, exports every declared symbol, host-side logic
(no compute calls; runs without a GPU)."""
import ctypes
import os
import re

import pytest

import fft_long_convolution_gb300 as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fftconv.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fftconv_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = F.lib()
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"
    assert sorted(F.EXPORTED) == names


def test_version_and_status_strings():
    assert F.lib().fftconv_version().decode().count(".") == 2
    for code in range(8):
        s = F.status_string(code)
        assert s and s != "unknown status"
    assert F.status_string(99) == "unknown status"


@pytest.mark.parametrize("N,R1", [(1024, 4), (2048, 8)])
def test_query_fused_factorization(N, R1):
    """Order 3 keeps the warp-level R1 x 16 x 16 kernel for N = 1024, 2048."""
    for dt in (F.F16, F.BF16):
        q = F.query(N, dt, order=3)
        assert q["path"] == F.PATH_FUSED and q["order"] == 3
        assert q["factors"] == [R1, 16, 16]
        assert q["factors"][0] * 16 * 16 == N == q["M"]
        assert q["kf_bytes_per_channel"] == 8 * N
        assert q["workspace_bytes_per_row"] == 0


@pytest.mark.parametrize("N", [8192, 16384, 32768])
def test_query_fused_tensor_core_factorization(N):
    """N = 8192, 16384 and 32768 (2N <= 64K) run fused as R0 x 64 x 64 (R0 =
    2, 4, 8) on the fifth-generation tensor cores; k_f holds one pass-B block
    (17 chunks of 4 warps x 2 halves x 32 lanes x 16 bytes) per pair of
    sub-rows."""
    for dt in (F.F16, F.BF16):
        q = F.query(N, dt)
        assert q["path"] == F.PATH_FUSED and q["order"] == 3
        assert q["factors"] == [N // 4096, 64, 64] and q["M"] == N
        assert q["kf_bytes_per_channel"] == (N // 8192) * 17 * 4 * 2 * 32 * 16
        assert q["workspace_bytes_per_row"] == 0


@pytest.mark.parametrize("N", [1024, 2048])
def test_query_short_rows_padded_to_4096(N):
    """By default N = 1024 and 2048 run on the 64 x 64 tensor-core kernel as
    rows zero-padded to 4096 (transform length M = 4096, 36 KB of k_f per
    channel); a frequency-sparse pattern keeps R1 x 16 x 16."""
    for dt in (F.F16, F.BF16):
        q = F.query(N, dt)
        assert q["path"] == F.PATH_FUSED and q["order"] == 2
        assert q["factors"] == [64, 64] and q["M"] == 4096 and q["N"] == N
        assert q["kf_bytes_per_channel"] == 9 * 4 * 2 * 32 * 16
        assert F.query(N, dt, order=2) == q
    assert F.sparse_query(N, F.BF16, [1, 1, 1]) == {"pairs_run": 0, "pairs_total": 0}


def test_query_fused_order2_4096():
    """N = 4096 runs as one 64 x 64 product on the fifth-generation tensor
    cores; its k_f holds 36 KB per channel (4096 bins plus zero padding bins
    in the kernel's column layout)."""
    for dt in (F.F16, F.BF16):
        q = F.query(4096, dt)
        assert q["path"] == F.PATH_FUSED and q["order"] == 2
        assert q["factors"] == [64, 64] and q["M"] == 4096
        assert q["kf_bytes_per_channel"] == 9 * 4 * 2 * 32 * 16
        assert q["workspace_bytes_per_row"] == 0


@pytest.mark.parametrize("N,R0", [(65536, 16), (262144, 64), (524288, 128)])
def test_query_multipass_order3_factorization(N, R0):
    """Sub-rows of 64 x 64 on the tensor cores: the default from N = 65536 up to 512K."""
    q = F.query(N, F.BF16)
    assert q["path"] == F.PATH_MULTIPASS and q["order"] == 3
    assert q["factors"] == [R0, 64, 64]
    assert R0 * 64 * 64 == N
    assert q["workspace_bytes_per_row"] == 4 * N
    # per pair of sub-rows: 17 chunks x 4 warps x 2 halves x 32 lanes x 16 bytes
    assert q["kf_bytes_per_channel"] == R0 // 2 * 17 * 4 * 2 * 32 * 16
    assert F.query(N, F.BF16, order=3) == q


@pytest.mark.parametrize("N,RA", [(1048576, 4), (2097152, 8)])
def test_query_multipass_two_level_factorization(N, RA):
    """Above N = 512K: the outer factor RA * 64 in two levels, sub-rows of 64 x 64."""
    q = F.query(N, F.BF16)
    assert q["path"] == F.PATH_MULTIPASS and q["order"] == 4
    assert q["factors"] == [RA, 64, 64, 64]
    assert RA * 64 * 64 * 64 == N
    assert q["workspace_bytes_per_row"] == 4 * N
    assert q["kf_bytes_per_channel"] == RA * 64 // 2 * 17 * 4 * 2 * 32 * 16
    assert F.query(N, F.BF16, order=4) == q


@pytest.mark.parametrize("N,R0,order", [(32768, 2, 4), (262144, 16, 4), (524288, 32, 4)])
def test_query_multipass_order4_factorization(N, R0, order):
    """Sub-rows of 64 x 16 x 16 on request up to N = 512K."""
    q = F.query(N, F.BF16, order=order)
    assert q["path"] == F.PATH_MULTIPASS and q["order"] == 4
    assert q["factors"] == [R0, 64, 16, 16]
    assert R0 * 64 * 16 * 16 == N
    assert q["workspace_bytes_per_row"] == 4 * N
    assert q["kf_bytes_per_channel"] == 8 * N


def test_query_multipass_order3_limit():
    with pytest.raises(F.FFTConvError) as e:
        F.query(1048576, F.BF16, order=3)
    assert e.value.status == 2


@pytest.mark.parametrize("N", [0, 1000, 512, 3 << 12, 1 << 22])
def test_query_rejects_unsupported_lengths(N):
    with pytest.raises(F.FFTConvError) as e:
        F.query(N, F.BF16)
    assert e.value.status == 2


def test_query_rejects_bad_order_and_dtype():
    with pytest.raises(F.FFTConvError):
        F.query(4096, F.BF16, order=3)
    with pytest.raises(F.FFTConvError):
        F.query(4096, 7)
    assert F.lib().fftconv_plan_query(4096, 1, 0, None) == 1


def test_null_plan_and_argument_validation_without_gpu():
    L = F.lib()
    vp = ctypes.c_void_p
    assert L.fftconv_forward(None, vp(16), vp(16), vp(16), 1, 1, None) == 1
    assert L.fftconv_forward_gated(None, vp(16), vp(16), vp(16), vp(16), vp(16), 1, 1, None) == 1
    assert L.fftconv_kernel_fft(None, vp(16), vp(16), 1, None) == 1
    assert L.fftconv_kf_bytes(None, 4) == 0
    assert L.fftconv_workspace_bytes(None, 1, 1) == 0
    assert L.fftconv_plan_destroy(None) == 0
    assert L.fftconv_set_workspace(None, None, 0) == 1
    h = ctypes.c_void_p()
    assert L.fftconv_plan_create(ctypes.byref(h), 1000, 1, 0) == 2 and not h.value
    assert L.fftconv_plan_create(None, 4096, 1, 0) == 1


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "fft_long_convolution_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle/" not in text and "liboracle" not in text, f


@pytest.mark.parametrize("C", [16384, 32768, 65536, 131072, 262144, 524288])
def test_circular_query_factorization(C):
    """A circular plan of length C transforms M = C/2 points as R0 x 64 x 64
    (R0 = C / 8192): C = 16384 on the fused kernel (no workspace), longer
    rows on the multi-pass path; its rows hold C samples."""
    for dt in (F.F16, F.BF16):
        q = F.circular_query(C, dt)
        R0 = C // 8192
        assert q["N"] == C and q["M"] == C // 2
        assert q["order"] == 3 and q["factors"] == [R0, 64, 64]
        if C == 16384:
            assert q["path"] == F.PATH_FUSED and q["workspace_bytes_per_row"] == 0
        else:
            assert q["path"] == F.PATH_MULTIPASS and q["workspace_bytes_per_row"] == 2 * C
        # the k_f of the causal plan with the same transform (pairs of 4096-point sub-rows)
        if C // 2 >= 65536:
            assert q["kf_bytes_per_channel"] == F.query(C // 2, dt)["kf_bytes_per_channel"]
        assert q["kf_bytes_per_channel"] == (R0 // 2) * 17 * 4 * 2 * 32 * 16


@pytest.mark.parametrize("C", [1024, 8192, 12288, 1 << 20, 0, -16384])
def test_circular_query_rejects_unsupported_lengths(C):
    with pytest.raises(F.FFTConvError) as e:
        F.circular_query(C, F.F16)
    assert e.value.status == 2
