"""Parity of the multi-pass CUDA path (N = 32K..2M) with the oracle (GPU)."""
import ctypes

import numpy as np
import pytest

import workloads as W
from _util import TOL, oracle_rows, rel_l2, run_gpu, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
F = pytest.importorskip("fft_long_convolution_gb300")


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("N,dtype,gated,B,H", [
    (65536, "fp16", False, 2, 3),
    (65536, "bf16", True, 1, 3),
    (65536, "bf16", False, 1, 2),
    (131072, "fp16", False, 1, 2),
    (262144, "bf16", True, 1, 2),
    (524288, "fp16", False, 1, 1),
    (1048576, "bf16", False, 1, 1),
    (1048576, "fp16", True, 2, 3),    # two-level RA = 4, gated, six rows
    (2097152, "bf16", False, 1, 1),
    (2097152, "fp16", True, 1, 2),    # two-level RA = 8, gated
])
def test_multipass_matches_oracle(N, dtype, gated, B, H):
    w = W.Workload("t", B, H, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=9)
    plan = F.Plan(N, torch_dtype(dtype))
    assert plan.info["path"] == F.PATH_MULTIPASS
    y, _ = run_gpu(plan, ins, gated)
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle_rows(ins, gated, threads=8)
    rel = rel_l2(got, ref)
    print(f"N={N} {dtype} gated={gated} rel-L2={rel:.3e} max-abs={np.abs(got - ref).max():.3e}")
    assert rel <= TOL[dtype]
    for b in range(B):
        for h in range(H):
            assert rel_l2(got[b, h], ref[b, h]) <= TOL[dtype]
    assert plan.device_status() == 0


@pytest.mark.parametrize("N,dtype,gated,B,H", [
    (32768, "bf16", True, 2, 2),
    (262144, "fp16", False, 1, 2),
])
def test_multipass_order4_matches_oracle(N, dtype, gated, B, H):
    """The 64 x 16 x 16 sub-rows on request at lengths whose default is 64 x 64."""
    w = W.Workload("t", B, H, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=11)
    plan = F.Plan(N, torch_dtype(dtype), order=4)
    assert plan.info["path"] == F.PATH_MULTIPASS and plan.info["order"] == 4
    y, _ = run_gpu(plan, ins, gated)
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle_rows(ins, gated, threads=8)
    rel = rel_l2(got, ref)
    print(f"order 4 N={N} {dtype} gated={gated} rel-L2={rel:.3e}")
    assert rel <= TOL[dtype]
    assert plan.device_status() == 0


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_multipass_delta_kernels(dtype):
    N, H = 65536, 4
    w = W.Workload("t", 1, H, N, dtype, False, "normal", "decay", "")
    ins = W.make_inputs(w, seed=10)
    shifts = [0, 1, N // 2, N - 1]
    k = np.zeros((H, N))
    for h, s in enumerate(shifts):
        k[h, s] = 1.0
    ins["k"] = W.round_to(k, "fp32")
    y, _ = run_gpu(F.Plan(N, torch_dtype(dtype)), ins, False)
    got = y.float().cpu().numpy().astype(np.float64)
    u = ins["u"].f64
    for h, s in enumerate(shifts):
        exp = np.zeros(N)
        exp[s:] = u[0, h, : N - s]
        un = np.linalg.norm(u[0, h])
        assert np.linalg.norm(got[0, h] - exp) <= TOL[dtype] * un, s
        assert np.abs(got[0, h, :s]).max(initial=0.0) <= 8 * TOL[dtype] * un / np.sqrt(N)


def test_multipass_needs_workspace():
    N = 65536
    plan = F.Plan(N, torch.bfloat16)
    assert plan.workspace_bytes(2, 3) == 2 * 3 * N * 4
    u = torch.zeros(2, 3, N, dtype=torch.bfloat16, device="cuda")
    kf = torch.zeros(plan.kf_bytes(3), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(u)
    L = F.lib()
    assert L.fftconv_forward(plan._h, u.data_ptr(), kf.data_ptr(), y.data_ptr(), 2, 3, None) == 4
    small = torch.empty(plan.workspace_bytes(2, 3) - 16, dtype=torch.uint8, device="cuda")
    plan.set_workspace(small)
    assert L.fftconv_forward(plan._h, u.data_ptr(), kf.data_ptr(), y.data_ptr(), 2, 3, None) == 4
    # a workspace overlapping the output is rejected
    big = torch.empty(plan.workspace_bytes(2, 3) + u.numel() * 2, dtype=torch.uint8, device="cuda")
    plan.set_workspace(big)
    yy = big[plan.workspace_bytes(2, 3) - 64:].view(torch.bfloat16)[: u.numel()].view(2, 3, N)
    assert L.fftconv_forward(plan._h, u.data_ptr(), kf.data_ptr(), yy.data_ptr(), 2, 3, None) == 1
    torch.cuda.synchronize()


@pytest.mark.parametrize("name,nrows", [("path512-256k", 6), ("gene-2m", 3)])
def test_workload_full_size_sampled(name, nrows):
    """The multi-pass workloads at full size, as the benchmark runs them;
    the oracle checks sampled rows."""
    w = W.WORKLOADS[name]
    ins = W.make_inputs(w, seed=0)
    plan = F.Plan(w.N, torch_dtype(w.dtype))
    y, _ = run_gpu(plan, ins, w.gated)
    rng = np.random.default_rng(12)
    flat = sorted(set([0, w.rows - 1] + list(rng.choice(w.rows, nrows - 2, replace=False))))
    ref = oracle_rows(ins, w.gated, rows=flat, threads=8).reshape(w.rows, w.N)
    got_all = y.view(w.rows, w.N)
    worst = 0.0
    for r in flat:
        g = got_all[r].float().cpu().numpy().astype(np.float64)
        rel = rel_l2(g, ref[r])
        worst = max(worst, rel)
        assert rel <= TOL[w.dtype], (r, rel)
    print(f"{name}: sampled rows {flat} worst rel-L2 {worst:.3e}")
    assert torch.isfinite(y.float()).all()
    assert plan.device_status() == 0


@pytest.mark.parametrize("N,dtype,gated,B,H", [
    (65536, "bf16", False, 3, 40),
    (65536, "fp16", True, 2, 40),
])
def test_multipass_many_items_every_row(N, dtype, gated, B, H):
    """Several work items per pipeline (next-item staging, pair changes,
    k_f prefetch) with every row compared with the oracle."""
    w = W.Workload("t", B, H, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=12)
    plan = F.Plan(N, torch_dtype(dtype))
    y, _ = run_gpu(plan, ins, gated)
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle_rows(ins, gated, threads=8)
    worst = max(rel_l2(got[b, h], ref[b, h]) for b in range(B) for h in range(H))
    print(f"N={N} {dtype} gated={gated} rows={B * H} worst row rel-L2={worst:.3e}")
    assert worst <= TOL[dtype]
    assert plan.device_status() == 0
