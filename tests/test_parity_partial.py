"""Parity of the partial convolution (kernel of at most W/2 taps over any
multiple of W/2) with the oracle (GPU)."""
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


@pytest.mark.parametrize("N,Wp,T,dtype,gated,B,H", [
    (16384, 4096, 2048, "bf16", False, 2, 3),     # tensor-memory kernel on the windows
    (16384, 4096, 700, "fp16", True, 1, 2),       # a kernel shorter than the half window
    (65536, 8192, 4096, "fp16", False, 1, 2),     # fused kernel on the windows
    (4194304, 2097152, 1048576, "bf16", False, 1, 1),  # N = 2^22 through multi-pass windows
])
def test_partial_matches_oracle(N, Wp, T, dtype, gated, B, H):
    w = W.Workload("t", B, H, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=41)
    k = ins["k"].f64[:, :T]
    plan = F.Plan(Wp, torch_dtype(dtype))
    kf = plan.kernel_fft_partial(torch.from_numpy(ins["k"].bits[:, :T].copy()).cuda())
    u = to_dev(ins["u"])
    if gated:
        y = plan.forward_partial(u, kf, to_dev(ins["w_in"]), to_dev(ins["w_out"]))
    else:
        y = plan.forward_partial(u, kf)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().astype(np.float64)
    x = ins["u"].f64 * (ins["w_in"].f64 if gated else 1.0)
    for b in range(B):
        for h in range(H):
            ref = oracle.partial_conv(x[b, h], k[h], T) * (ins["w_out"].f64[b, h] if gated else 1.0)
            rel = rel_l2(got[b, h], ref)
            assert rel <= TOL[dtype], (b, h, rel)
    print(f"partial N={N} W={Wp} T={T} {dtype} gated={gated} last rel-L2={rel:.3e}")
    assert plan.device_status() == 0


def test_partial_argument_errors():
    plan = F.Plan(4096, torch.bfloat16)
    L = F.lib()
    u = torch.zeros(1, 1, 3000, dtype=torch.bfloat16, device="cuda")
    kf = torch.zeros(plan.kf_bytes(1), dtype=torch.uint8, device="cuda")
    assert L.fftconv_partial_scratch_bytes(plan._h, 1, 1, 3000, 0) == 0  # not a multiple of 2048
    assert L.fftconv_forward_partial(plan._h, u.data_ptr(), None, None, kf.data_ptr(), u.data_ptr(), 1, 1, 3000,
                                     None, 0, None) in (1, 2)
    u = torch.zeros(1, 1, 4096, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(u)
    assert L.fftconv_forward_partial(plan._h, u.data_ptr(), None, None, kf.data_ptr(), y.data_ptr(), 1, 1, 4096,
                                     None, 0, None) == 4
    with pytest.raises(ValueError):
        plan.kernel_fft_partial(torch.zeros(1, 2049, device="cuda"))
