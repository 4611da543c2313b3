"""Parity of the backward pass (input and kernel gradients) with the oracle (GPU)."""
import numpy as np
import pytest

import workloads as W
from _util import TOL, rel_l2, to_dev, torch_dtype

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
F = pytest.importorskip("fft_long_convolution_gb300")


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(B, H, N, dtype, gated, seed):
    w = W.Workload("t", B, H, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=seed)
    # the output gradient: another seeded 16-bit tensor of u's shape
    dy = W.make_inputs(W.Workload("t", B, H, N, dtype, False, "normal", "decay", ""), seed=seed + 1000)["u"]
    return ins, dy


@pytest.mark.parametrize("N,dtype,gated,B,H,order", [
    (1024, "fp16", False, 2, 3, 0),
    (4096, "bf16", True, 3, 4, 0),
    (8192, "fp16", True, 2, 2, 0),
    (16384, "bf16", False, 1, 3, 0),
    (65536, "fp16", False, 1, 2, 0),
    (65536, "bf16", True, 2, 1, 4),
])
def test_input_grad_matches_oracle(N, dtype, gated, B, H, order):
    ins, dy = _inputs(B, H, N, dtype, gated, seed=31)
    plan = F.Plan(N, torch_dtype(dtype), order=order)
    kfa = plan.kernel_fft_adjoint(to_dev(ins["k"]))
    if gated:
        du = plan.backward_du(to_dev(dy), kfa, to_dev(ins["w_in"]), to_dev(ins["w_out"]))
        ref = oracle.input_grad_batch(dy.f64, ins["k"].f64, ins["w_in"].f64, ins["w_out"].f64, threads=8)
    else:
        du = plan.backward_du(to_dev(dy), kfa)
        ref = oracle.input_grad_batch(dy.f64, ins["k"].f64, threads=8)
    torch.cuda.synchronize()
    got = du.float().cpu().numpy().astype(np.float64)
    rel = rel_l2(got, ref)
    print(f"du N={N} {dtype} gated={gated} rel-L2={rel:.3e}")
    assert rel <= TOL[dtype]
    for b in range(B):
        for h in range(H):
            assert rel_l2(got[b, h], ref[b, h]) <= 2 * TOL[dtype]
    assert plan.device_status() == 0


@pytest.mark.parametrize("N,dtype,gated,B,H", [
    (1024, "fp16", False, 3, 2),      # shared-memory channels
    (4096, "bf16", True, 4, 3),
    (4096, "fp16", False, 1, 5),
    (8192, "fp16", True, 2, 2),       # four-step, L = 8 x 2048
    (16384, "fp16", True, 3, 2),      # four-step, L = 16 x 2048
    (16384, "bf16", False, 1, 3),
    (32768, "bf16", False, 2, 2),     # four-step, L = 32 x 2048
    (65536, "fp16", False, 1, 2),     # four-step with the columns through HBM, L = 64 x 2048
    (131072, "bf16", True, 2, 1),     # L = 128 x 2048
    (262144, "fp16", False, 1, 2),    # L = 256 x 2048 (the path512 length)
    (524288, "bf16", False, 1, 1),    # L = 512 x 2048
    (1048576, "fp16", False, 1, 1),   # L = 1024 x 2048 (tiles of 8 columns)
    (2097152, "bf16", True, 1, 1),    # L = 2048 x 2048 (tiles of 4 columns), the longest plan
])
def test_kernel_grad_matches_oracle(N, dtype, gated, B, H):
    ins, dy = _inputs(B, H, N, dtype, gated, seed=32)
    plan = F.Plan(N, torch_dtype(dtype))
    u = to_dev(ins["u"])
    if gated:
        dk = plan.backward_dk(u, to_dev(dy), to_dev(ins["w_in"]), to_dev(ins["w_out"]))
        ref = oracle.kernel_grad(ins["u"].f64, dy.f64, ins["w_in"].f64, ins["w_out"].f64, threads=8)
    else:
        dk = plan.backward_dk(u, to_dev(dy))
        ref = oracle.kernel_grad(ins["u"].f64, dy.f64, threads=8)
    torch.cuda.synchronize()
    got = dk.cpu().numpy().astype(np.float64)
    rel = rel_l2(got, ref)
    print(f"dk N={N} {dtype} gated={gated} rel-L2={rel:.3e}")
    # the inputs are the same rounded values; only float32 transform rounding remains
    assert rel <= 1e-4


def test_gradients_are_adjoints_on_device():
    """<forward(u), dy> = <u, du> and = <k, dk> up to 16-bit rounding."""
    B, H, N = 2, 3, 4096
    ins, dy = _inputs(B, H, N, "bf16", False, seed=33)
    plan = F.Plan(N, torch.bfloat16)
    k = to_dev(ins["k"])
    u, d = to_dev(ins["u"]), to_dev(dy)
    y = plan.forward(u, plan.kernel_fft(k)).double()
    du = plan.backward_du(d, plan.kernel_fft_adjoint(k)).double()
    dk = plan.backward_dk(u, d).double()
    lhs = float((y * d.double()).sum())
    assert abs(lhs - float((u.double() * du).sum())) <= 1e-2 * float((u.double() * du).abs().sum())
    assert abs(lhs - float((k.double() * dk).sum())) <= 1e-2 * float((k.double() * dk).abs().sum())


def test_kernel_grad_edge_cases():
    plan = F.Plan(1024, torch.float16)
    L = F.lib()
    dk = torch.full((2, 1024), 7.0, device="cuda")
    assert L.fftconv_backward_dk(plan._h, None, None, None, None, dk.data_ptr(), 0, 2, None, 0, None) == 0
    torch.cuda.synchronize()
    assert float(dk.abs().max()) == 0.0  # B = 0: zero gradient
    # 2N <= 8192: whole channels in shared memory, no scratch
    assert L.fftconv_backward_dk_scratch_bytes(plan._h, 1, 2) == 0
    big = F.Plan(8192, torch.float16)
    u = torch.zeros(1, 2, 8192, dtype=torch.float16, device="cuda")
    dk8 = torch.empty(2, 8192, device="cuda")
    need = L.fftconv_backward_dk_scratch_bytes(big._h, 1, 2)
    assert need == 2 * 16384 * 8  # four-step form: the per-channel inverse intermediate
    assert L.fftconv_backward_dk(big._h, u.data_ptr(), u.data_ptr(), None, None, dk8.data_ptr(), 1, 2, None, 0,
                                 None) == 4
