"""Tensor-core decode on fp8 caches with queries far from N(0,1), against the
oracle within the fp8 tolerance.

With an fp8 cache the tensor-core decode multiplies the cache's e4m3 codes
as stored, so the queries enter its MMAs as two e4m3 terms after a power of
two chosen per (sequence, KV head) from the largest |q| of the G query rows.
These cases move that choice to its edges: every query tiny (scale 2^-12),
every query large (scores with a standard deviation near 8, a sharp
softmax), query heads of one KV head spread over 2^16 in magnitude, and rows
whose queries are all zero (the scale's zero case: uniform weights).  The
cache write, and so the codes, are those of the other fp8 tests ("Inside
vLLM v0.7", "FP8 KV cache"); only q changes."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import paged_kv_cache_writes_gb300 as pa
from paged_kv_cache_writes_gb300.staging import DeviceBatch, to_bits
from _gpu import TOL, max_err, oracle_pools

pytestmark = pytest.mark.gpu

LENS = [1, 17, 130, 300, 512, 513, 1000, 2049]


def _transform(q_bits, src, kind, G):
    q = W.bits_to_f32(q_bits, src).astype(np.float64)
    if kind == "tiny":
        q = q * 2.0 ** -12
    elif kind == "sharp":
        q = q * 8.0
    elif kind == "spread":
        h = np.arange(q.shape[1]) % G
        q = q * (2.0 ** (-8.0 + 16.0 * h / (G - 1)))[None, :, None]
    elif kind == "zero_rows":
        q = q.copy()
        q[0] = 0.0
        q[3] = 0.0
    return W.round_to_bits(q.astype(np.float32), src)


@pytest.mark.parametrize("kind", ["tiny", "sharp", "spread", "zero_rows"])
@pytest.mark.parametrize("src", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (64, 8, 32), (64, 4, 16)])
def test_fp8_decode_query_range(kind, src, hq, hkv, bs):
    b = W.decode_batch("qrange", LENS, hq, hkv, 128, bs, src, kv_dtype="fp8", seed=hq + 3 * hkv + bs,
                       partition_size=512)
    b.q = _transform(b.q, src, kind, hq // hkv)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.step_all()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kp, vp = oracle_pools(b)
    assert np.array_equal(to_bits(dev.k_cache), kp) and np.array_equal(to_bits(dev.v_cache), vp)
    ref = oracle.decode_batch(b, kp, vp)
    err = max_err(dev.out, ref)
    assert err <= TOL["fp8"], err
