"""Helpers for the GPU parity tests: run a seeded batch through the C ABI
(via the package's staging helper) and through the oracle, on the same inputs."""
import numpy as np
import torch

import oracle
import workloads as W

TOL = {"f16": 2e-3, "bf16": 2e-3, "fp8": 2e-2}


def run_gpu(b, step=True, out_dtype="f32"):
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    import paged_kv_cache_writes_gb300 as pa
    dev = DeviceBatch(b, "cuda", out_dtype=out_dtype)
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
    """max |gpu - oracle| for an fp32 GPU output (the accumulation result)."""
    assert got.dtype == torch.float32
    g = got.cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), "non-finite GPU output"
    return float(np.abs(g - ref).max()) if g.size else 0.0


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half the spacing of ``dtype`` values at magnitude x (its RNE storage error bound)."""
    mant, emin = {"bf16": (8, -126), "f16": (11, -14)}[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** emin)))
    return 2.0 ** (np.maximum(e, emin) - mant)


def rounded_excess(got: torch.Tensor, ref: np.ndarray, dtype: str, tol: float) -> float:
    """For an output stored in a 16-bit dtype: the error beyond the allowance
    tol + half an ulp of the stored magnitude (<= 0 means within bounds)."""
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), "non-finite GPU output"
    allow = tol + half_ulp(np.abs(ref) + tol, dtype)
    return float((np.abs(g - ref) - allow).max()) if g.size else 0.0
