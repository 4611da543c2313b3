"""Failure detection without a GPU fault: a bounded on-device wait on a phase
that nothing completes gives up, the plan's error word reports it, and the
context keeps working (GPU)."""
import time

import numpy as np
import pytest

import workloads as W
from _util import TOL, oracle_rows, rel_l2, run_gpu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
F = pytest.importorskip("fft_long_convolution_gb300")


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("sleep", [0, 1])
def test_bounded_wait_gives_up_and_is_reported(sleep):
    plan = F.Plan(4096, torch.bfloat16)
    L = F.lib()
    assert plan.device_status() == 0
    t0 = time.perf_counter()
    assert L.fftconv_selftest_wait(plan._h, sleep, None) == 0
    status = plan.device_status()  # synchronises
    dt = time.perf_counter() - t0
    print(f"sleep={sleep}: gave up after {dt:.3f} s")
    assert status == 7  # FFTCONV_ERR_TIMEOUT
    assert dt < 5.0  # each wait is bounded to about one second of wall time
    assert plan.device_status() == 0  # reading cleared it
    # the context still runs the real path correctly
    w = W.Workload("t", 2, 2, 4096, "bf16", True, "normal", "decay", "")
    ins = W.make_inputs(w, seed=61)
    y, _ = run_gpu(plan, ins, True)
    got = y.float().cpu().numpy().astype(np.float64)
    assert rel_l2(got, oracle_rows(ins, True)) <= TOL["bf16"]
    assert plan.device_status() == 0
