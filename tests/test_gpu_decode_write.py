"""The fused decode step (pa_decode_write): each sequence's new token stored at
its last position's slot, then paged decode with it included, in one call.

Checked against the oracle's own cache write and decode on the same inputs
(outputs within the decode tolerance; cache contents bit for bit), on the
tensor-core kernel (where the decode launch stores the token) and on the
CUDA-core kernel (a cache-write launch, then decode)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_writes_gb300 as pa
import workloads as W
from paged_kv_cache_writes_gb300.staging import DeviceBatch, to_bits
from _gpu import TOL, max_err, oracle_pools

pytestmark = pytest.mark.gpu

LENS = [1, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1000, 1537, 0, 4100]


def _fused(b, kernel="auto"):
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    with pa.decode_kernel(kernel):
        dev.decode_write()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kp, vp = oracle_pools(b)   # the oracle's pools after its own step write
    assert np.array_equal(to_bits(dev.k_cache), kp) and np.array_equal(to_bits(dev.v_cache), vp)
    ref = oracle.decode_batch(b, kp, vp)
    err = max_err(dev.out, ref)
    assert err <= TOL[b.kv_dtype], err
    return dev


@pytest.mark.parametrize("kernel", ["auto", "cuda_cores"])
@pytest.mark.parametrize("kv,src", [("bf16", "bf16"), ("f16", "f16"), ("fp8", "bf16"), ("fp8", "f16")])
@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (64, 8, 32), (32, 2, 16)])
def test_fused_step_matches_write_then_decode(kernel, kv, src, hq, hkv, bs):
    b = W.decode_batch("fused", LENS, hq, hkv, 128, bs, src, kv_dtype=kv, seed=hq + hkv * 3 + bs, partition_size=512)
    _fused(b, kernel)


@pytest.mark.parametrize("kernel", ["auto", "cuda_cores"])
@pytest.mark.parametrize("kv", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (16, 2, 32)])
def test_fused_step_head_dim_64(kernel, kv, hq, hkv, bs):
    b = W.decode_batch("fused d64", LENS, hq, hkv, 64, bs, kv, seed=hq + hkv + bs + 64, partition_size=512)
    _fused(b, kernel)


@pytest.mark.parametrize("kernel", ["auto", "cuda_cores"])
@pytest.mark.parametrize("q", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (64, 8, 32)])
def test_fused_step_head_dim_64_fp8(kernel, q, hq, hkv, bs):
    # 64-byte cache rows: the new token's eight 8-code chunks per row, and no store past the row
    b = W.decode_batch("fused d64 fp8", LENS, hq, hkv, 64, bs, q, kv_dtype="fp8", seed=hq + hkv + bs + 65,
                       partition_size=512)
    _fused(b, kernel)


@pytest.mark.parametrize("ps", [32, 96, 0])
def test_fused_step_partition_sizes(ps):
    b = W.decode_batch("fused ps", [1, 40, 700, 2049, 3000], 16, 2, 128, 16, "bf16", seed=51, partition_size=ps)
    _fused(b)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_fused_step_llama70b_full(kv):
    # the benchmark's step on its workload: cache bit for bit, every output row against the oracle
    _fused(W.cfg_llama70b(kv_dtype=kv))


def test_fused_step_equals_separate_calls_bitwise():
    """Stored bytes and outputs of the fused call equal those of the write and decode as two calls."""
    b = W.decode_batch("fused eq", LENS, 32, 8, 128, 16, "bf16", seed=52, partition_size=512)
    a = DeviceBatch(b, "cuda")
    a.run_setup()
    a.decode_write()
    c = DeviceBatch(b, "cuda")
    c.run_setup()
    c.write_step()
    c.decode()
    torch.cuda.synchronize()
    assert torch.equal(a.k_cache.view(torch.int16), c.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), c.v_cache.view(torch.int16))
    assert torch.equal(a.out.view(torch.int32), c.out.view(torch.int32))


def test_fused_step_rejects_a_slot_other_than_the_last_position():
    b = W.decode_batch("fused bad", [40, 70], 32, 8, 128, 16, "bf16", seed=53)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    k, v, slots = dev.fused_step_tensors()
    bad = slots.clone()
    bad[1] = slots[1] - 1                       # an earlier position of the same row
    before = dev.k_cache.clone()
    pa.pa_decode_write(dev.q, k, v, bad, dev.k_cache, dev.v_cache, dev.desc, dev.block_tables, dev.seq_lens,
                       int(b.seq_lens.max()), b.scale, dev.out, dev.workspace, b.partition_size)
    assert pa.pa_get_device_error() == 4        # PA_ERR_DEVICE_CHECK
    blk, off = int(bad[1]) // 16, int(bad[1]) % 16
    assert torch.equal(dev.k_cache[blk, :, off].view(torch.int16), before[blk, :, off].view(torch.int16))
