"""Parity of frequency-sparse plans with the oracle's masked convolution
(GPU): fused lengths (pattern applied through k_f), the multi-pass lengths
with pairs of sub-rows skipped (one and two HBM levels, both pass-B
engines), the degenerate patterns, and a sampled full-size check."""
import numpy as np
import pytest

import oracle
import workloads as W
from _util import TOL, rel_l2, run_gpu, to_dev, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
F = pytest.importorskip("fft_long_convolution_gb300")


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _oracle(ins, mask, gated, rows=None):
    return oracle.masked_causal_conv_batch(ins["u"].f64, ins["k"].f64, mask,
                                           ins["w_in"].f64 if gated else None,
                                           ins["w_out"].f64 if gated else None, threads=8, rows=rows)


def _check(N, dtype, gated, B, H, band, order=0, seed=21, u_kind="normal", k_kind="decay"):
    w = W.Workload("t", B, H, N, dtype, gated, u_kind, k_kind, "")
    ins = W.make_inputs(w, seed=seed)
    plan = F.Plan(N, torch_dtype(dtype), order=order, band=band)
    info = plan.info
    mask = oracle.band_mask(N, info["factors"], band)
    bd = plan.band()
    assert bd["band"] == [min(b, Mj // 2 + 1) for b, Mj in zip(band, info["factors"])]
    q = F.sparse_query(N, plan.dtype, band, order)
    assert (bd["pairs_run"], bd["pairs_total"]) == (q["pairs_run"], q["pairs_total"])
    y, _ = run_gpu(plan, ins, gated)
    got = y.float().cpu().numpy().astype(np.float64).reshape(B * H, N)
    ref = _oracle(ins, mask, gated)
    rel = rel_l2(got, ref)
    print(f"N={N} {dtype} gated={gated} band={band} kept={mask[:N].mean():.3f} "
          f"pairs {bd['pairs_run']}/{bd['pairs_total']} rel-L2={rel:.3e}")
    assert rel <= TOL[dtype]
    for r in range(B * H):
        assert rel_l2(got[r], ref[r]) <= TOL[dtype]
    assert plan.device_status() == 0
    return bd


@pytest.mark.parametrize("N,dtype,gated,B,H,band", [
    (1024, "fp16", False, 2, 3, [2, 5, 8]),
    (4096, "bf16", True, 2, 3, [9, 20]),
    (4096, "fp16", False, 1, 2, [33, 3]),
    (16384, "fp16", False, 1, 3, [20, 9, 9]),
    (16384, "bf16", False, 2, 3, [1, 33, 33]),       # outer digit 0 only: pair (1, 3) not run
    (16384, "fp16", True, 1, 3, [1, 20, 9]),         # and the inner axes cut
    (16384, "bf16", True, 2, 2, [2, 12, 33]),        # digits 0, +-1 kept: both pairs run
    (8192, "fp16", False, 1, 2, [1, 33, 20]),
    (32768, "bf16", False, 1, 2, [3, 20, 20]),
])
def test_fused_sparse(N, dtype, gated, B, H, band):
    bd = _check(N, dtype, gated, B, H, band)
    if N >= 8192:  # the fused tensor-core kernel: pairs of sub-rows (k0, R0 - k0)
        R0 = N // 4096
        assert bd["pairs_total"] == R0 // 2
        assert bd["pairs_run"] == (1 if (R0 == 4 and band[0] <= 1) else R0 // 2)
    else:
        assert bd["pairs_total"] == 0


@pytest.mark.parametrize("N,dtype,gated,B,H,band", [
    (65536, "fp16", False, 2, 3, [3, 33, 33]),        # outer digits 0, +-1, +-2 kept
    (65536, "bf16", True, 1, 3, [5, 20, 33]),
    (262144, "bf16", False, 1, 2, [16, 33, 33]),      # half of the pairs skipped
    (262144, "fp16", True, 1, 2, [9, 20, 7]),         # all three axes cut
    (524288, "bf16", False, 1, 1, [40, 33, 12]),      # R0 = 128
])
def test_multipass_sparse_skips_pairs(N, dtype, gated, B, H, band):
    bd = _check(N, dtype, gated, B, H, band)
    assert 0 < bd["pairs_run"] < bd["pairs_total"]


@pytest.mark.parametrize("N,dtype,gated,B,H,band", [
    (1048576, "bf16", False, 1, 1, [2, 16, 33, 33]),   # two HBM levels: first-level digits 0, +-1 of 4
    (2097152, "bf16", False, 1, 1, [5, 9, 33, 20]),
    (2097152, "fp16", False, 1, 1, [1, 33, 33, 33]),   # first-level digit 0 only: 32 of 256 pairs run
    (1048576, "fp16", True, 2, 3, [2, 9, 33, 33]),     # gated, six rows; live runs of 9 and 8 rows per k_a
    (2097152, "bf16", True, 1, 2, [8, 5, 33, 33]),     # every k_a live, runs of 5 and 4 rows
])
def test_two_level_sparse(N, dtype, gated, B, H, band):
    """The fused outer passes of a two-level plan skip dead sub-rows: pass A
    does not store them and pass C reads them as zeros (pass B never writes
    them)."""
    bd = _check(N, dtype, gated, B, H, band)
    assert 0 < bd["pairs_run"] < bd["pairs_total"]


@pytest.mark.parametrize("N,band", [(65536, [1, 20, 9, 9]), (262144, [5, 33, 4, 9])])
def test_order4_warp_level_pass_b_sparse(N, band):
    bd = _check(N, "bf16", True, 2, 2, band, order=4)
    assert 0 < bd["pairs_run"] < bd["pairs_total"]


@pytest.mark.parametrize("N,band", [(4096, [0, 33]), (262144, [0, 33, 33]), (262144, [33, 0, 33]),
                                    (2097152, [5, 33, 0, 33])])
def test_empty_pattern_gives_zero(N, band):
    w = W.Workload("t", 1, 2, N, "bf16", True, "normal", "decay", "")
    ins = W.make_inputs(w, seed=3)
    plan = F.Plan(N, torch.bfloat16, band=band)
    if plan.info["path"] == F.PATH_MULTIPASS:
        assert plan.band()["pairs_run"] == 0
    y, _ = run_gpu(plan, ins, True)
    assert torch.count_nonzero(y).item() == 0
    assert plan.device_status() == 0


@pytest.mark.parametrize("N", [4096, 262144])
def test_full_band_equals_dense_plan(N):
    w = W.Workload("t", 1, 2, N, "bf16", False, "normal", "decay", "")
    ins = W.make_inputs(w, seed=4)
    dense = F.Plan(N, torch.bfloat16)
    full = F.Plan(N, torch.bfloat16, band=[Mj // 2 + 1 for Mj in dense.info["factors"]])
    yd, _ = run_gpu(dense, ins, False)
    yf, _ = run_gpu(full, ins, False)
    assert torch.equal(yd, yf)  # bitwise: nothing is masked or skipped


def test_sparse_plan_rejects_unsupported_calls():
    plan = F.Plan(262144, torch.bfloat16, band=[16, 33, 33])
    L = F.lib()
    assert L.fftconv_backward_dk(plan._h, None, None, None, None, None, 1, 1, None, 0, None) == 2
    assert L.fftconv_forward_circular(plan._h, None, None, None, None, None, 1, 1, None, 0, None) == 2
    assert L.fftconv_forward_partial(plan._h, None, None, None, None, None, 1, 1, 1024, None, 0, None) == 2


def test_full_size_gene_sampled():
    """gene-2m recipe at full length (H = 4 channels of the one-hot input),
    75 % of the pairs skipped; two rows checked against the oracle in full."""
    N, band = 2097152, [3, 16, 33, 33]
    w = W.scaled(W.WORKLOADS["gene-2m"], H=4)
    ins = W.make_inputs(w, seed=0)
    plan = F.Plan(N, torch.bfloat16, band=band)
    bd = plan.band()
    assert 0 < bd["pairs_run"] < bd["pairs_total"]
    y, _ = run_gpu(plan, ins, False)
    got = y.float().cpu().numpy().astype(np.float64).reshape(4, N)
    mask = oracle.band_mask(N, plan.info["factors"], band)
    ref = _oracle(ins, mask, False, rows=[0, 3])
    for i, r in enumerate([0, 3]):
        rel = rel_l2(got[r], ref[i])
        print(f"gene-2m row {r}: pairs {bd['pairs_run']}/{bd['pairs_total']} rel-L2={rel:.3e}")
        assert rel <= TOL["bf16"]
    assert plan.device_status() == 0


@pytest.mark.parametrize("N,dtype,gated,B,H,band", [
    (4096, "bf16", True, 2, 3, [9, 20]),
    (16384, "fp16", False, 1, 2, [20, 9, 9]),
    (262144, "bf16", False, 1, 2, [16, 33, 33]),
    (1048576, "bf16", False, 1, 1, [2, 16, 33, 33]),
])
def test_sparse_input_grad(N, dtype, gated, B, H, band):
    """du of the frequency-sparse convolution: a forward with the adjoint k_f
    of the same sparse plan (skipped pairs included) against the oracle's
    masked correlation."""
    w = W.Workload("t", B, H, N, dtype, gated, "normal", "decay", "")
    ins = W.make_inputs(w, seed=41)
    dy = W.make_inputs(W.Workload("t", B, H, N, dtype, False, "normal", "decay", ""), seed=1041)["u"]
    plan = F.Plan(N, torch_dtype(dtype), band=band)
    mask = oracle.band_mask(N, plan.info["factors"], band)
    kfa = plan.kernel_fft_adjoint(to_dev(ins["k"]))
    if gated:
        du = plan.backward_du(to_dev(dy), kfa, to_dev(ins["w_in"]), to_dev(ins["w_out"]))
        ref = oracle.masked_input_grad_batch(dy.f64, ins["k"].f64, mask, ins["w_in"].f64, ins["w_out"].f64,
                                             threads=8)
    else:
        du = plan.backward_du(to_dev(dy), kfa)
        ref = oracle.masked_input_grad_batch(dy.f64, ins["k"].f64, mask, threads=8)
    torch.cuda.synchronize()
    got = du.float().cpu().numpy().astype(np.float64)
    rel = rel_l2(got, ref)
    print(f"sparse du N={N} {dtype} gated={gated} band={band} rel-L2={rel:.3e}")
    assert rel <= TOL[dtype]
    assert plan.device_status() == 0
