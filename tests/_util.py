"""Shared helpers of the GPU tests: move seeded inputs to the device, run the
CUDA path through the C ABI, and compare with the oracle."""
import numpy as np

import oracle
import workloads as W

TOL = {"fp16": 2e-3, "bf16": 1e-2}  # rel-L2 bars for 16-bit inputs


def torch_dtype(dtype):
    import torch
    return torch.float16 if dtype == "fp16" else torch.bfloat16


def to_dev(r, dtype=None, device="cuda"):
    import torch
    if r.dtype == "fp32":
        return torch.from_numpy(np.ascontiguousarray(r.bits)).to(device)
    return torch.from_numpy(np.ascontiguousarray(r.bits).view(np.int16)).view(torch_dtype(r.dtype)).to(device)


def rel_l2(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def run_gpu(plan, ins, gated):
    """k_f and y through the C ABI for the given rounded inputs."""
    import torch
    kf = plan.kernel_fft(to_dev(ins["k"]))
    u = to_dev(ins["u"])
    if gated:
        y = plan.forward_gated(u, to_dev(ins["w_in"]), to_dev(ins["w_out"]), kf)
    else:
        y = plan.forward(u, kf)
    torch.cuda.synchronize()
    return y, kf


def oracle_rows(ins, gated, rows=None, threads=8):
    """Oracle output (double) for all rows or for the listed flat row ids."""
    return oracle.causal_conv_batch(ins["u"].f64, ins["k"].f64,
                                    ins["w_in"].f64 if gated else None,
                                    ins["w_out"].f64 if gated else None,
                                    threads=threads, rows=rows)
