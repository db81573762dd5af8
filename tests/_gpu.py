"""Helpers for the GPU parity tests: run a seeded batch through the C ABI
(via the package's staging helper) and through the oracle, on the same inputs."""
import numpy as np
import torch

import oracle
import workloads as W

TOL = {"f16": 2e-3, "bf16": 2e-3, "fp8": 2e-2}


def run_gpu(b, step=True):
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    import paged_kv_cache_writes_gb300 as pa
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    if step:
        dev.step_all()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    return dev


def oracle_pools(b, step=True):
    kp, vp = W.empty_pools(b)
    oracle.populate(b, kp, vp, step=step)
    return kp, vp


def max_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.float().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite GPU output"
    return float(np.abs(g - ref).max()) if g.size else 0.0
