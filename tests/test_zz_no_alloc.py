"""The no-allocation forward entry point (GPU).

fftconv_forward_noalloc serves callers that cannot allocate device memory
(for example code living inside a framework whose allocator owns the GPU, or
a plug-in that only receives its input and output buffers): it keeps the
multi-pass intermediate in a fixed array inside the library instead of a
caller workspace.  It runs the same kernels as fftconv_forward on the same
inputs, so these tests require bitwise equality with it (two calls in a row,
the array keeping the first call's contents), and check one case against
the oracle.  The file name makes pytest collect it last.
"""
import numpy as np
import pytest

import workloads as W
from _util import TOL, oracle_rows, rel_l2, to_dev, torch_dtype

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


def _noalloc(plan, u, kf, B, H):
    y = torch.full_like(u, float("nan"))
    stream = torch.cuda.current_stream().cuda_stream
    st = F.lib().fftconv_forward_noalloc(plan._h, u.data_ptr(), kf.data_ptr(), y.data_ptr(), B, H, stream)
    assert st == 0, F.status_string(st)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("N,dtype", [(65536, "bf16"), (32768, "fp16"), (4096, "bf16"), (16384, "fp16")])
def test_noalloc_matches_forward_bitwise_on_two_calls(N, dtype):
    B, H = 2, 3
    ins = _inputs(N, dtype, B, H, seed=21)
    plan = F.Plan(N, torch_dtype(dtype))
    kf = plan.kernel_fft(to_dev(ins["k"]))
    u = to_dev(ins["u"])
    ref = plan.forward(u, kf)  # existing entry point (caller workspace on multi-pass lengths)
    torch.cuda.synchronize()
    for _ in range(2):
        y = _noalloc(plan, u, kf, B, H)
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    # and against the oracle, at the bar of the input dtype
    got = y.float().cpu().numpy().astype(np.float64)
    rel = rel_l2(got, oracle_rows(ins, False))
    assert rel <= TOL[dtype], rel
    assert plan.device_status() == 0


@pytest.mark.parametrize("C", [16384, 65536])
def test_noalloc_circular_plan_matches_forward_bitwise(C):
    """A circular plan's rows (C samples; the fused kernel at 16384, the
    multi-pass intermediate of C/2 complex points above) through the fixed array."""
    B, H = 2, 3
    ins = _inputs(C, "bf16", B, H, seed=24)
    plan = F.Plan(C, torch.bfloat16, circular=True)
    kf = plan.kernel_fft(to_dev(ins["k"]))
    u = to_dev(ins["u"])
    ref = plan.forward(u, kf)
    torch.cuda.synchronize()
    y = _noalloc(plan, u, kf, B, H)
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
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
    torch.cuda.synchronize()


def test_noalloc_largest_call_that_fits():
    """The largest call that fits the array (N = 2^21, 8 rows: the two-level
    multi-pass path over all 64 MiB) on random inputs and a real kernel
    spectrum, after earlier calls left data in the array: bitwise equal to
    the forward with a caller workspace."""
    N = 2097152
    Hmax = SCRATCH_BYTES // (4 * N)
    ins = _inputs(N, "bf16", 1, Hmax, seed=23)
    plan = F.Plan(N, torch.bfloat16)
    assert plan.workspace_bytes(1, Hmax) == SCRATCH_BYTES
    kf = plan.kernel_fft(to_dev(ins["k"]))
    u = to_dev(ins["u"])
    ref = plan.forward(u, kf)
    torch.cuda.synchronize()
    y = _noalloc(plan, u, kf, 1, Hmax)
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    # one row against the oracle in full
    ref3 = oracle_rows(ins, False, rows=[3])[0, 3]
    got3 = y[0, 3].float().cpu().numpy().astype(np.float64)
    assert rel_l2(got3, ref3) <= TOL["bf16"]
    assert plan.device_status() == 0
