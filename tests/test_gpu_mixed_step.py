"""pa_mixed_step on the GPU: a chunked-prefill batch and a decode batch of
one layer in one call ("Inside vLLM v0.7", "Architectural Blueprint 3:
Chunked Prefill"), against the oracle.

Where both parts run on the tensor cores (head_dim 128, 4 or 8 query heads
per KV head) the call is one launch after the decode's plan: prefill tiles
and decode CTAs share a grid.  Other shapes, and the CUDA-core decode, take
two launches.  Either way the decode output must equal pa_decode's bit for
bit (the same units, merged in the same order) and both outputs must match
the oracle within the tolerance of the cache dtype; with the decode rows'
new tokens stored by the call itself the cache must equal the oracle's
bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_writes_gb300 as pa
import workloads as W
from paged_kv_cache_writes_gb300.staging import DeviceBatch, to_bits
from _gpu import TOL, max_err, oracle_pools

pytestmark = pytest.mark.gpu


def _batch(src, kv, hq, hkv, d, bs, seed, chunk=200, q_start=300, num_decode=12, dec_max=1500):
    return W.mixed_prefill_batch("mixed step", chunk=chunk, q_start=q_start, num_decode=num_decode, dec_min=1,
                                 dec_max=dec_max, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                                 src_dtype=src, kv_dtype=kv, seed=seed)


def _check(dev, b):
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kp, vp = oracle_pools(b)
    assert np.array_equal(to_bits(dev.k_cache), kp) and np.array_equal(to_bits(dev.v_cache), vp)
    err_d = max_err(dev.out, oracle.decode_batch(b, kp, vp))
    err_p = max_err(dev.prefill["out"], oracle.prefill_batch(b, kp, vp))
    assert err_d <= TOL[b.kv_dtype], err_d
    assert err_p <= TOL[b.kv_dtype], err_p


# one launch: G = 4 or 8, head_dim 128; two launches: G = 16, head_dim 64
SHAPES = [("bf16", "fp8", 32, 8, 128, 16), ("f16", "fp8", 64, 8, 128, 32), ("bf16", "bf16", 32, 8, 128, 16),
          ("f16", "f16", 64, 8, 128, 32), ("bf16", "bf16", 64, 4, 128, 16), ("bf16", "fp8", 8, 4, 64, 16)]


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("src,kv,hq,hkv,d,bs", SHAPES)
def test_mixed_step_against_the_oracle(src, kv, hq, hkv, d, bs, fused):
    b = _batch(src, kv, hq, hkv, d, bs, seed=hq + hkv + d + bs + fused)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.mixed_step(fused=fused)
    _check(dev, b)


@pytest.mark.parametrize("kernel", ["auto", "cuda_cores"])
def test_mixed_step_decode_equals_pa_decode(kernel):
    b = _batch("bf16", "fp8", 32, 8, 128, 16, seed=7, num_decode=20, dec_max=3000)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.write_step()
    with pa.decode_kernel(kernel):
        dev.decode()
        alone = dev.out.clone()
        dev.out.zero_()
        dev.mixed_attention()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert torch.equal(dev.out, alone)
    kp, vp = oracle_pools(b)
    assert max_err(dev.prefill["out"], oracle.prefill_batch(b, kp, vp)) <= TOL["fp8"]


def test_mixed_step_with_an_empty_part():
    b = _batch("bf16", "bf16", 32, 8, 128, 16, seed=9)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.write_step()
    p = dev.prefill
    dev.decode()
    dec_alone = dev.out.clone()
    dev.prefill_chunk()
    pre_alone = p["out"].clone()
    dev.out.zero_()
    p["out"].zero_()
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    # prefill part empty: the decode alone
    pa.pa_mixed_step(dev.q, dev.block_tables, dev.seq_lens, int(b.seq_lens.max()), dev.out, p["q"], z, z[:0], 0,
                     p["block_tables"], p["seq_lens"][:0], 0, p["out"], dev.k_cache, dev.v_cache, dev.desc, b.scale,
                     dev.workspace)
    # decode part empty: the prefill alone
    pa.pa_mixed_step(dev.q[:0], dev.block_tables[:0], dev.seq_lens[:0], 0, dev.out[:0], p["q"], p["cu_q_lens"],
                     p["q_start"], p["max_q_len"], p["block_tables"], p["seq_lens"], p["max_seq_len"], p["out"],
                     dev.k_cache, dev.v_cache, dev.desc, b.scale)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert torch.equal(dev.out, dec_alone) and torch.equal(p["out"], pre_alone)


def test_mixed_step_at_full_size():
    # the chunked-prefill mixed batch: one 512-row chunk at 4096 + 128 decodes (256..8192 tokens), fp8 KV
    b = W.cfg_mixed_fp8()
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.mixed_step(fused=True)
    _check(dev, b)
