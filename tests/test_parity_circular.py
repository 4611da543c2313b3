"""Parity of the circular (non-causal) convolution with the oracle (GPU)."""
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


@pytest.mark.parametrize("C,dtype,gated,B,H", [
    (512, "fp16", False, 2, 3),       # plan 1024 (fused)
    (2048, "bf16", True, 3, 2),       # plan 4096 (tensor-memory kernel)
    (8192, "fp16", False, 1, 2),      # plan 16384 (fused, 4 x 64 x 64 on the tensor cores)
    (65536, "bf16", False, 1, 2),     # plan 131072 (multi-pass)
])
def test_circular_matches_oracle(C, dtype, gated, B, H):
    w = W.Workload("t", B, H, C, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=51)
    plan = F.Plan(2 * C, torch_dtype(dtype))
    kf = plan.kernel_fft_partial(torch.from_numpy(ins["k"].bits.copy()).cuda())
    u = to_dev(ins["u"])
    if gated:
        y = plan.forward_circular(u, kf, to_dev(ins["w_in"]), to_dev(ins["w_out"]))
    else:
        y = plan.forward_circular(u, kf)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().astype(np.float64)
    x = ins["u"].f64 * (ins["w_in"].f64 if gated else 1.0)
    for b in range(B):
        for h in range(H):
            ref = oracle.circular_conv(x[b, h], ins["k"].f64[h]) * (ins["w_out"].f64[b, h] if gated else 1.0)
            rel = rel_l2(got[b, h], ref)
            assert rel <= TOL[dtype], (b, h, rel)
    print(f"circular C={C} {dtype} gated={gated} last rel-L2={rel:.3e}")
    assert plan.device_status() == 0


def test_circular_shift_wraps_on_device():
    """k = delta_s: y = u rolled by s (the end of the row reappears at the start)."""
    C, H = 2048, 3
    plan = F.Plan(2 * C, torch.float16)
    shifts = [1, 1000, C - 1]
    k = torch.zeros(H, C, device="cuda")
    for h, s in enumerate(shifts):
        k[h, s] = 1.0
    u = torch.randn(1, H, C, device="cuda").half()
    y = plan.forward_circular(u, plan.kernel_fft_partial(k))
    torch.cuda.synchronize()
    for h, s in enumerate(shifts):
        exp = torch.roll(u[0, h].float(), s)
        assert float((y[0, h].float() - exp).norm() / exp.norm()) <= TOL["fp16"]


@pytest.mark.parametrize("C,dtype,gated,B,H", [
    (16384, "fp16", True, 2, 3),      # R0 = 2, fused: one pair of sub-rows
    (16384, "bf16", False, 3, 1),     # fused, an odd row count (one pipeline idle at the end)
    (16384, "fp16", False, 4, 101),   # fused, 404 rows: several rows per CTA
    (16384, "bf16", True, 2, 161),    # fused gated, 322 rows
    (32768, "bf16", False, 1, 3),     # R0 = 4
    (65536, "bf16", True, 1, 2),      # R0 = 8
    (131072, "fp16", False, 2, 1),    # R0 = 16
    (524288, "bf16", False, 1, 1),    # R0 = 64, the largest
])
def test_native_circular_matches_oracle(C, dtype, gated, B, H):
    """The circular plan: C samples per row, k of C taps, all outer rows in
    and out (no zero padding, no truncation)."""
    w = W.Workload("t", B, H, C, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=52)
    plan = F.Plan(C, torch_dtype(dtype), circular=True)
    assert plan.info["N"] == C and plan.info["M"] == C // 2
    kf = plan.kernel_fft(torch.from_numpy(ins["k"].bits.copy()).cuda())
    u = to_dev(ins["u"])
    if gated:
        y = plan.forward_gated(u, to_dev(ins["w_in"]), to_dev(ins["w_out"]), kf)
    else:
        y = plan.forward(u, kf)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().astype(np.float64)
    x = ins["u"].f64 * (ins["w_in"].f64 if gated else 1.0)
    for b in range(B):
        for h in range(H):
            ref = oracle.circular_conv(x[b, h], ins["k"].f64[h]) * (ins["w_out"].f64[b, h] if gated else 1.0)
            rel = rel_l2(got[b, h], ref)
            assert rel <= TOL[dtype], (b, h, rel)
    print(f"native circular C={C} {dtype} gated={gated} last rel-L2={rel:.3e}")
    assert plan.device_status() == 0


@pytest.mark.parametrize("C", [16384, 32768])
def test_native_circular_shift_and_adjoint(C):
    """k = delta_s rolls each row by s; the adjoint k_f gives the circular
    correlation, i.e. the convolution with the reversed kernel k[-m mod C]."""
    H = 3
    plan = F.Plan(C, torch.float16, circular=True)
    shifts = [1, 12345, C - 1]
    k = torch.zeros(H, C, device="cuda")
    for h, s in enumerate(shifts):
        k[h, s] = 1.0
    u = torch.randn(2, H, C, device="cuda").half()
    y = plan.forward(u, plan.kernel_fft(k))
    torch.cuda.synchronize()
    for b in range(2):
        for h, s in enumerate(shifts):
            exp = torch.roll(u[b, h].float(), s)
            assert float((y[b, h].float() - exp).norm() / exp.norm()) <= TOL["fp16"]
    w = W.Workload("t", 1, 2, C, "bf16", False, "normal", "decay", "")
    ins = W.make_inputs(w, seed=53)
    planb = F.Plan(C, torch.bfloat16, circular=True)
    kfa = planb.kernel_fft_adjoint(torch.from_numpy(ins["k"].bits.copy()).cuda())
    du = planb.backward_du(to_dev(ins["u"]), kfa)
    torch.cuda.synchronize()
    got = du.float().cpu().numpy().astype(np.float64)
    for h in range(2):
        krev = np.roll(ins["k"].f64[h][::-1], 1)  # k[-m mod C]
        ref = oracle.circular_conv(ins["u"].f64[0, h], krev)
        assert rel_l2(got[0, h], ref) <= TOL["bf16"]
    assert plan.device_status() == 0 and planb.device_status() == 0


def test_native_circular_rejects_other_calls():
    plan = F.Plan(16384, torch.float16, circular=True)
    L = F.lib()
    u = torch.zeros(1, 1, 16384, dtype=torch.float16, device="cuda")
    dk = torch.empty(1, 16384, device="cuda")
    # kernel gradient and the windowed forms are not defined on a circular plan
    assert L.fftconv_backward_dk(plan._h, u.data_ptr(), u.data_ptr(), None, None, dk.data_ptr(), 1, 1, None, 0,
                                 None) == 2
    assert L.fftconv_forward_circular(plan._h, u.data_ptr(), None, None, u.data_ptr(), u.data_ptr(), 1, 1, None, 0,
                                      None) == 2
