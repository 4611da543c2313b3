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
