"""fp8 caches with one scale per KV head on the GPU, against the oracle
(which reads per-head scales as the per-tensor rule applied head by head):
cache bytes bit for bit after the write, decode on both kernels and the fused
step, prefill on both kernels, within the fp8 tolerance."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_writes_gb300 as pa
import workloads as W
from paged_kv_cache_writes_gb300.staging import DeviceBatch, to_bits
from _gpu import TOL, max_err, oracle_pools

pytestmark = pytest.mark.gpu

LENS = [1, 17, 33, 300, 512, 513, 1000, 2049]


@pytest.mark.parametrize("kernel", ["auto", "cuda_cores"])
@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv,d,bs", [(32, 8, 128, 16), (64, 8, 128, 32), (8, 4, 64, 16)])
def test_decode_with_per_head_scales(kernel, src, hq, hkv, d, bs):
    b = W.decode_batch("hs", LENS, hq, hkv, d, bs, src, kv_dtype="fp8", seed=hq + hkv + d + bs,
                       partition_size=512, fp8_scales="head")
    assert len(set(np.asarray(b.k_scale).tolist())) > 1
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    with pa.decode_kernel(kernel):
        dev.step_all()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kp, vp = oracle_pools(b)
    assert np.array_equal(to_bits(dev.k_cache), kp) and np.array_equal(to_bits(dev.v_cache), vp)
    err = max_err(dev.out, oracle.decode_batch(b, kp, vp))
    assert err <= TOL["fp8"], err


def test_fused_step_with_per_head_scales():
    b = W.decode_batch("hsf", LENS, 32, 8, 128, 16, "bf16", kv_dtype="fp8", seed=61, fp8_scales="head")
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.decode_write()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kp, vp = oracle_pools(b)
    assert np.array_equal(to_bits(dev.k_cache), kp) and np.array_equal(to_bits(dev.v_cache), vp)
    assert max_err(dev.out, oracle.decode_batch(b, kp, vp)) <= TOL["fp8"]


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 4, 64), (12, 4, 128)])
def test_prefill_with_per_head_scales(hq, hkv, d):
    # head_dim 128 with 8 query heads per KV head runs on the tensor cores; the others on CUDA cores
    b = W.prefill_batch("hsp", [(300, 200), (0, 77), (1000, 129)], hq, hkv, d, 16, "bf16", kv_dtype="fp8",
                        seed=62 + hq, fp8_scales="head")
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.step_all()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kp, vp = oracle_pools(b)
    ref = oracle.prefill_batch(b, kp, vp)
    err = max_err(dev.prefill["out"], ref)
    assert err <= TOL["fp8"], err
