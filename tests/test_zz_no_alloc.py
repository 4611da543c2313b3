"""The no-allocation forward entry point (GPU).

fftconv_forward_noalloc serves callers that cannot allocate device memory
(for example code living inside a framework whose allocator owns the GPU, or
a plug-in that only receives its input and output buffers): it keeps the
multi-pass intermediate in a fixed array inside the library instead of a
caller workspace.  These tests call it through the C ABI and compare it with
fftconv_forward, which uses a caller workspace, on two calls in a row.  The
file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

import workloads as W
from _util import TOL, rel_l2, to_dev, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
F = pytest.importorskip("fft_long_convolution_gb300")

SCRATCH_BYTES = 64 << 20  # FFTCONV_STATIC_SCRATCH_BYTES


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(N, dtype, B, H, seed):
    w = W.Workload("t", B, H, N, dtype, False, "normal", "decay", "")
    return W.make_inputs(w, seed=seed)


@pytest.mark.parametrize("N,dtype", [(65536, "bf16"), (32768, "fp16"), (4096, "bf16")])
def test_noalloc_matches_forward_on_two_calls(N, dtype):
    B, H = 2, 3
    ins = _inputs(N, dtype, B, H, seed=21)
    plan = F.Plan(N, torch_dtype(dtype))
    kf = plan.kernel_fft(to_dev(ins["k"]))
    u = to_dev(ins["u"])
    ref = plan.forward(u, kf)  # existing entry point (caller workspace on multi-pass lengths)
    torch.cuda.synchronize()
    ref64 = ref.float().cpu().numpy().astype(np.float64)
    L = F.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        y = torch.full_like(u, float("nan"))
        st = L.fftconv_forward_noalloc(plan._h, u.data_ptr(), kf.data_ptr(), y.data_ptr(), B, H, stream)
        assert st == 0, F.status_string(st)
        torch.cuda.synchronize()
        got = y.float().cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert rel_l2(got, ref64) <= TOL[dtype]
    assert plan.device_status() == 0


def test_noalloc_rejects_calls_beyond_the_scratch_size():
    N = 2097152
    plan = F.Plan(N, torch.bfloat16)
    B, H = 1, SCRATCH_BYTES // (4 * N) + 1  # one row more than the array holds
    assert plan.workspace_bytes(B, H) > SCRATCH_BYTES
    u = torch.zeros(B, H, N, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(u)
    kf = torch.zeros(plan.kf_bytes(H), dtype=torch.uint8, device="cuda")
    st = F.lib().fftconv_forward_noalloc(plan._h, u.data_ptr(), kf.data_ptr(), y.data_ptr(), B, H, None)
    assert st == 4  # FFTCONV_ERR_WORKSPACE, nothing launched
    # the largest call that fits is accepted
    Hmax = SCRATCH_BYTES // (4 * N)
    st = F.lib().fftconv_forward_noalloc(plan._h, u.data_ptr(), kf.data_ptr(), y.data_ptr(), B, Hmax, None)
    assert st == 0
    torch.cuda.synchronize()
