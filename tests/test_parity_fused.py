"""Parity of the fused CUDA path with the oracle (GPU)."""
import numpy as np
import pytest

import workloads as W
from _util import TOL, oracle_rows, rel_l2, run_gpu, to_dev, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
F = pytest.importorskip("fft_long_convolution_gb300")

FUSED_N = [1024, 2048, 4096, 8192, 16384, 32768]


def _plan(N, dtype):
    return F.Plan(N, torch_dtype(dtype))


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("N", FUSED_N)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("gated", [False, True])
def test_fused_matches_oracle(N, dtype, gated):
    # B*H = 15 rows: a ragged tail for every rows-per-CTA packing (1, 2, 4)
    w = W.Workload("t", 3, 5, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=3)
    plan = _plan(N, dtype)
    y, _ = run_gpu(plan, ins, gated)
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle_rows(ins, gated)
    rel = rel_l2(got, ref)
    print(f"N={N} {dtype} gated={gated} rel-L2={rel:.3e} max-abs={np.abs(got - ref).max():.3e}")
    assert rel <= TOL[dtype]
    # every row individually within the bar (no row left unwritten)
    for r in range(w.rows):
        b, h = divmod(r, w.H)
        assert rel_l2(got[b, h], ref[b, h]) <= 2 * TOL[dtype]
    assert plan.device_status() == 0


@pytest.mark.parametrize("N", [1024, 4096, 8192, 16384, 32768])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_delta_kernels(N, dtype):
    """k = delta_s gives y[t] = u[t-s] (t >= s): pins causal truncation.

    The rounding error of an FFT convolution scales with |u|*|k| (Parseval),
    not with |y|; for s = N-1 the output has one nonzero sample, so the error
    is bounded relative to the input norm here."""
    H = 4
    w = W.Workload("t", 2, H, N, dtype, False, "normal", "decay", "")
    ins = W.make_inputs(w, seed=5)
    shifts = [0, 1, N // 2, N - 1]
    k = np.zeros((H, N))
    for h, s in enumerate(shifts):
        k[h, s] = 1.0
    ins["k"] = W.round_to(k, "fp32")
    y, _ = run_gpu(_plan(N, dtype), ins, False)
    got = y.float().cpu().numpy().astype(np.float64)
    u = ins["u"].f64
    for b in range(2):
        for h, s in enumerate(shifts):
            exp = np.zeros(N)
            exp[s:] = u[b, h, : N - s]
            un = np.linalg.norm(u[b, h])
            assert np.linalg.norm(got[b, h] - exp) <= TOL[dtype] * un, (b, h, s)
            # causal: nothing before the shift beyond the rounding floor
            assert np.abs(got[b, h, :s]).max(initial=0.0) <= 8 * TOL[dtype] * un / np.sqrt(N)


def test_u_delta_returns_kernel():
    N, H = 4096, 3
    w = W.Workload("t", 1, H, N, "fp16", False, "normal", "normal_scaled", "")
    ins = W.make_inputs(w, seed=6)
    u = np.zeros((1, H, N))
    u[:, :, 0] = 1.0
    ins["u"] = W.round_to(u, "fp16")
    y, _ = run_gpu(_plan(N, "fp16"), ins, False)
    got = y.float().cpu().numpy()[0].astype(np.float64)
    assert rel_l2(got, ins["k"].f64) <= TOL["fp16"]


def test_deterministic_and_empty():
    N = 4096
    w = W.Workload("t", 2, 7, N, "bf16", True, "normal", "decay", "")
    ins = W.make_inputs(w, seed=7)
    plan = _plan(N, "bf16")
    y1, kf = run_gpu(plan, ins, True)
    y2, _ = run_gpu(plan, ins, True)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    # B*H = 0 launches nothing and succeeds
    e = torch.empty(0, 7, N, dtype=torch.bfloat16, device="cuda")
    plan.forward(e, kf, y=torch.empty_like(e))


def test_validation_on_device_buffers():
    N = 1024
    plan = _plan(N, "fp16")
    u = torch.zeros(2, 2, N, dtype=torch.float16, device="cuda")
    kf = torch.zeros(plan.kf_bytes(2), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(u)
    L = F.lib()
    # misaligned pointer -> ALIGN
    assert L.fftconv_forward(plan._h, u.data_ptr() + 2, kf.data_ptr(), y.data_ptr(), 1, 2, None) == 3
    # y overlapping u -> INVALID
    assert L.fftconv_forward(plan._h, u.data_ptr(), kf.data_ptr(), u.data_ptr(), 2, 2, None) == 1
    # NULL k_f -> INVALID
    assert L.fftconv_forward(plan._h, u.data_ptr(), None, y.data_ptr(), 2, 2, None) == 1
    # negative sizes -> INVALID
    assert L.fftconv_forward(plan._h, u.data_ptr(), kf.data_ptr(), y.data_ptr(), -1, 2, None) == 1
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["causal-1k", "hyena-gated-4k", "m2bert-16k"])
def test_workload_full_size_sampled(name):
    """Full-size workloads in the launch configuration the benchmark times;
    the oracle checks a sample of rows (all rows for the 1K case)."""
    w = W.WORKLOADS[name]
    ins = W.make_inputs(w, seed=0)
    plan = _plan(w.N, w.dtype)
    y, _ = run_gpu(plan, ins, w.gated)
    rng = np.random.default_rng(11)
    flat = list(range(w.rows)) if w.rows <= 64 else sorted(
        set([0, w.rows - 1] + list(rng.choice(w.rows, 30, replace=False))))
    ref = oracle_rows(ins, w.gated, rows=flat).reshape(w.rows, w.N)
    got_all = y.view(w.rows, w.N)
    rels = []
    for r in flat:
        g = got_all[r].float().cpu().numpy().astype(np.float64)
        rels.append(rel_l2(g, ref[r]))
        assert rels[-1] <= TOL[w.dtype], (r, rels[-1])
    print(f"{name}: sampled rows {len(flat)} worst rel-L2 {max(rels):.3e}")
    assert torch.isfinite(y.float()).all()
    assert plan.device_status() == 0


@pytest.mark.parametrize("dtype,gated", [("bf16", True), ("fp16", False)])
def test_tc64_many_items_every_row(dtype, gated):
    """N = 4096 with several row pairs per pipeline and an odd batch (the
    last pair of every channel has no second row); every row checked."""
    w = W.Workload("t", 7, 180, 4096, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=13)
    plan = _plan(4096, dtype)
    y, _ = run_gpu(plan, ins, gated)
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle_rows(ins, gated, threads=8)
    worst = max(rel_l2(got[b, h], ref[b, h]) for b in range(w.B) for h in range(w.H))
    print(f"N=4096 {dtype} gated={gated} rows={w.rows} worst row rel-L2={worst:.3e}")
    assert worst <= TOL[dtype]
    assert plan.device_status() == 0


@pytest.mark.parametrize("N,dtype,gated", [(16384, "fp16", False), (16384, "bf16", True),
                                           (8192, "bf16", False), (8192, "fp16", True),
                                           (32768, "bf16", False), (32768, "fp16", True)])
def test_ftc_many_rows_every_row(N, dtype, gated):
    """N = 8192 / 16384 / 32768 on the fused tensor-core kernel with several
    rows per pipeline (the next row's staging overlaps the current row; pair
    (1, 3) hands its outputs to pair (0, 2); for 32768 the two pipelines pass
    the accumulator and the staging between them); every row checked."""
    w = W.Workload("t", 5, 130, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=17)
    plan = _plan(N, dtype)
    y, _ = run_gpu(plan, ins, gated)
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle_rows(ins, gated, threads=8)
    worst = max(rel_l2(got[b, h], ref[b, h]) for b in range(w.B) for h in range(w.H))
    print(f"N={N} {dtype} gated={gated} rows={w.rows} worst row rel-L2={worst:.3e}")
    assert worst <= TOL[dtype]
    assert plan.device_status() == 0


@pytest.mark.parametrize("N", [1024, 2048])
@pytest.mark.parametrize("dtype,gated", [("fp16", False), ("bf16", True)])
def test_short_rows_order3_warp_level_kernel(N, dtype, gated):
    """N = 1024 / 2048 with order 3: the warp-level R1 x 16 x 16 kernel
    (the default pads these rows to 4096 on the tensor cores)."""
    w = W.Workload("t", 3, 5, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=19)
    plan = F.Plan(N, torch_dtype(dtype), order=3)
    assert plan.info["order"] == 3 and plan.info["factors"][1] == 16
    y, _ = run_gpu(plan, ins, gated)
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle_rows(ins, gated)
    assert rel_l2(got, ref) <= TOL[dtype]
    assert plan.device_status() == 0


@pytest.mark.parametrize("N,B,H", [(1024, 7, 37), (2048, 3, 50)])
def test_short_rows_padded_every_row(N, B, H):
    """N = 1024 / 2048 on the 4096-point tensor-core kernel (rows zero-padded
    in shared memory, only outputs t < N stored): several row pairs per
    pipeline, an odd batch, every row checked, and nothing written beyond the
    rows."""
    w = W.Workload("t", B, H, N, "bf16", True, "normal", "decay", "")
    ins = W.make_inputs(w, seed=23)
    plan = _plan(N, "bf16")
    assert plan.info["order"] == 2 and plan.info["M"] == 4096
    kf = plan.kernel_fft(to_dev(ins["k"]))
    u, wi, wo = to_dev(ins["u"]), to_dev(ins["w_in"]), to_dev(ins["w_out"])
    guard = torch.full((B * H * N + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = guard[: B * H * N].view(B, H, N)
    plan.forward_gated(u, wi, wo, kf, y=y)
    torch.cuda.synchronize()
    assert torch.all(guard[B * H * N:] == 7.0)
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle_rows(ins, True, threads=8)
    worst = max(rel_l2(got[b, h], ref[b, h]) for b in range(B) for h in range(H))
    assert worst <= TOL["bf16"], worst
    assert plan.device_status() == 0
