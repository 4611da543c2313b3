"""fftconv_forward_host: host-resident rows through the chunked copy /
convolution pipeline give the device path's results bit for bit (GPU)."""
import ctypes

import numpy as np
import pytest

import workloads as W
from _util import TOL, oracle_rows, rel_l2, to_dev, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
F = pytest.importorskip("fft_long_convolution_gb300")


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _host(r, tdt, pinned=True):
    t = torch.from_numpy(r.bits.view(np.int16)).view(tdt)
    return t.pin_memory() if pinned else t.clone()


@pytest.mark.parametrize("N,dtype,gated,B,H,order", [
    (1024, "fp16", False, 2, 8, 0),       # fused, two chunks of one batch entry
    (4096, "bf16", True, 7, 20, 0),       # tensor-memory kernel, seven chunks: buffer sets reused
    (16384, "fp16", False, 9, 5, 0),      # fused, chunks of two batch entries and a short last one
    (65536, "bf16", False, 1, 12, 0),     # multi-pass 64 x 64, B = 1: chunks of channels (k_f offsets)
    (32768, "bf16", False, 1, 12, 0),     # fused 8 x 64 x 64, B = 1: chunks of channels (k_f offsets)
    (65536, "fp16", True, 3, 2, 4),       # multi-pass 64 x 16 x 16
])
def test_host_matches_device(N, dtype, gated, B, H, order):
    w = W.Workload("t", B, H, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=21)
    tdt = torch_dtype(dtype)
    plan = F.Plan(N, tdt, order=order)
    kf = plan.kernel_fft(to_dev(ins["k"]))
    u = to_dev(ins["u"])
    if gated:
        y_dev = plan.forward_gated(u, to_dev(ins["w_in"]), to_dev(ins["w_out"]), kf)
        y_host = plan.forward_host(_host(ins["u"], tdt), kf, _host(ins["w_in"], tdt), _host(ins["w_out"], tdt))
    else:
        y_dev = plan.forward(u, kf)
        y_host = plan.forward_host(_host(ins["u"], tdt), kf)
    torch.cuda.synchronize()
    assert not y_host.is_cuda
    assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
    assert plan.device_status() == 0


@pytest.mark.parametrize("C,dtype,gated,B,H", [
    (16384, "bf16", True, 2, 5),      # circular plan on the fused kernel
    (32768, "fp16", True, 3, 4),      # circular plan, chunks of batch entries
    (65536, "bf16", False, 1, 6),     # circular plan, B = 1: chunks of channels
])
def test_host_matches_device_circular(C, dtype, gated, B, H):
    """The host-buffer call on a circular plan (rows of C samples)."""
    w = W.Workload("t", B, H, C, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=23)
    tdt = torch_dtype(dtype)
    plan = F.Plan(C, tdt, circular=True)
    kf = plan.kernel_fft(to_dev(ins["k"]))
    if gated:
        y_dev = plan.forward_gated(to_dev(ins["u"]), to_dev(ins["w_in"]), to_dev(ins["w_out"]), kf)
        y_host = plan.forward_host(_host(ins["u"], tdt), kf, _host(ins["w_in"], tdt), _host(ins["w_out"], tdt))
    else:
        y_dev = plan.forward(to_dev(ins["u"]), kf)
        y_host = plan.forward_host(_host(ins["u"], tdt), kf)
    torch.cuda.synchronize()
    assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
    assert plan.device_status() == 0


def test_host_pageable_memory_and_oracle():
    """Pageable host memory serialises the copies but gives the same rows."""
    w = W.Workload("t", 4, 6, 4096, "bf16", False, "normal", "decay", "")
    ins = W.make_inputs(w, seed=22)
    tdt = torch.bfloat16
    plan = F.Plan(4096, tdt)
    kf = plan.kernel_fft(to_dev(ins["k"]))
    y = torch.empty(w.B, w.H, w.N, dtype=tdt)
    plan.forward_host(_host(ins["u"], tdt, pinned=False), kf, y=y)
    torch.cuda.synchronize()
    got = y.float().numpy().astype(np.float64)
    assert rel_l2(got, oracle_rows(ins, False)) <= TOL["bf16"]


def test_host_argument_errors():
    N, B, H = 4096, 2, 3
    plan = F.Plan(N, torch.bfloat16)
    L = F.lib()
    u = torch.zeros(B, H, N, dtype=torch.bfloat16).pin_memory()
    y = torch.zeros_like(u).pin_memory()
    kf = torch.zeros(plan.kf_bytes(H), dtype=torch.uint8, device="cuda")
    need = L.fftconv_host_scratch_bytes(plan._h, B, H, 0)
    assert need > 0 and L.fftconv_host_scratch_bytes(plan._h, B, H, 1) > need
    scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
    call = lambda *a: L.fftconv_forward_host(plan._h, *a)
    assert call(u.data_ptr(), None, None, kf.data_ptr(), y.data_ptr(), B, H, scratch.data_ptr(), need - 256, None) == 4
    assert call(u.data_ptr(), None, None, kf.data_ptr(), y.data_ptr(), B, H, None, 0, None) == 4
    assert call(u.data_ptr(), u.data_ptr(), None, kf.data_ptr(), y.data_ptr(), B, H, scratch.data_ptr(), need,
                None) == 1
    assert call(u.data_ptr(), None, None, kf.data_ptr(), u.data_ptr(), B, H, scratch.data_ptr(), need, None) == 1
    assert call(u.data_ptr(), None, None, kf.data_ptr() + 4, y.data_ptr(), B, H, scratch.data_ptr(), need,
                None) == 3
    assert call(u.data_ptr(), None, None, kf.data_ptr(), y.data_ptr(), 0, H, None, 0, None) == 0
    assert call(u.data_ptr(), None, None, kf.data_ptr(), y.data_ptr(), B, H, scratch.data_ptr(), need, None) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("N,dtype,B,H,band", [
    (262144, "bf16", 3, 2, [16, 33, 33]),       # one-level sparse passes, chunks of batch entries
    (1048576, "bf16", 1, 3, [2, 16, 33, 33]),   # two-level sparse passes, chunks of channels
])
def test_host_sparse_plan_matches_device(N, dtype, B, H, band):
    """A frequency-sparse plan through the chunked host pipeline: each chunk
    restarts the row index, which must not move the skipped sub-rows."""
    w = W.Workload("t", B, H, N, dtype, False, "normal", "decay", "")
    ins = W.make_inputs(w, seed=23)
    tdt = torch_dtype(dtype)
    plan = F.Plan(N, tdt, band=band)
    assert 0 < plan.band()["pairs_run"] < plan.band()["pairs_total"]
    kf = plan.kernel_fft(to_dev(ins["k"]))
    y_dev = plan.forward(to_dev(ins["u"]), kf)
    y_host = plan.forward_host(_host(ins["u"], tdt), kf)
    torch.cuda.synchronize()
    assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
    assert plan.device_status() == 0
