"""GPU parity of chunked-prefill attention against the fp64 oracle.

Row r of a chunk at absolute position q_start + r attends causally to
positions 0 .. q_start + r of its sequence.  Every batch is compared on every
row, head and element, including the chunk of the chunked-prefill mixed batch
and each prefill batch the benchmark times.

head_dim 128 with a GQA group of 1, 2, 4, 8 or 16 runs on the tensor-core
kernel (128 GQA-packed rows per Q tile, 128-key tiles); head_dim 64 and other
groups run on the CUDA-core row kernel.  Both are covered here."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _gpu import TOL, max_err, oracle_pools, rounded_excess, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("src,kv", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "fp8")])
@pytest.mark.parametrize("hq,hkv,d,bs", [(32, 8, 128, 16), (8, 8, 64, 32), (16, 2, 128, 32)])
def test_prefill_small(src, kv, hq, hkv, d, bs):
    chunks = [(0, 37), (100, 64), (17, 1), (512, 130), (31, 33)]
    b = W.prefill_batch("p", chunks, hq, hkv, d, bs, src, kv_dtype=kv, seed=hq + d + bs)
    dev = run_gpu(b)
    kp, vp = oracle_pools(b)
    ref = oracle.prefill_batch(b, kp, vp)
    assert max_err(dev.prefill["out"], ref) <= TOL[kv]


def test_prefill_query_dtype_output():
    b = W.prefill_batch("p", [(0, 37), (100, 64)], 32, 8, 128, 16, "bf16", seed=9)
    dev = run_gpu(b, out_dtype="q")
    kp, vp = oracle_pools(b)
    ref = oracle.prefill_batch(b, kp, vp)
    assert rounded_excess(dev.prefill["out"], ref, "bf16", TOL["bf16"]) <= 0


def test_mixed_fp8_prefill_full():
    # the chunk of the chunked-prefill mixed batch (512 rows at 4096, fp8 KV), every row, and its decode part
    b = W.cfg_mixed_fp8()
    dev = run_gpu(b)
    kp, vp = oracle_pools(b)
    assert max_err(dev.prefill["out"], oracle.prefill_batch(b, kp, vp)) <= TOL["fp8"]
    assert max_err(dev.out, oracle.decode_batch(b, kp, vp)) <= TOL["fp8"]


@pytest.mark.parametrize("key", sorted(W.PREFILL_WORKLOADS))
def test_benchmarked_prefill_batches_full(key):
    # each prefill batch the benchmark times, at its full size, every row
    b = W.PREFILL_WORKLOADS[key][1]()
    dev = run_gpu(b)
    kp, vp = oracle_pools(b)
    err = max_err(dev.prefill["out"], oracle.prefill_batch(b, kp, vp))
    assert err <= TOL[b.kv_dtype], err


def test_prefill_seq_len_mismatch_sets_error():
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    b = W.prefill_batch("p", [(20, 10)], 8, 8, 64, 16, "bf16", seed=5)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.write_step()
    dev.prefill["seq_lens"][0] += 1
    dev.prefill_chunk()
    assert pa.pa_get_device_error() == 4


# chunks that cross the 128-packed-row CTA boundary for every group size, a
# chunk of one row at position 0, an empty chunk, and contexts that end
# inside a 64-key tile and inside a block
RAGGED_CHUNKS = [(0, 1), (0, 77), (45, 0), (300, 129), (1000, 8), (63, 65)]


@pytest.mark.parametrize("src,kv", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "fp8"), ("f16", "fp8")])
@pytest.mark.parametrize("hq,hkv,bs", [(8, 8, 16), (16, 8, 32), (64, 8, 16), (32, 2, 16)])
def test_prefill_tensor_core_groups(src, kv, hq, hkv, bs):
    b = W.prefill_batch("p", RAGGED_CHUNKS, hq, hkv, 128, bs, src, kv_dtype=kv, seed=hq * 3 + hkv + bs)
    dev = run_gpu(b)
    kp, vp = oracle_pools(b)
    ref = oracle.prefill_batch(b, kp, vp)
    assert max_err(dev.prefill["out"], ref) <= TOL[kv]


def test_prefill_uneven_group_uses_row_kernel():
    # GQA group 3 at head_dim 128: the CUDA-core path
    b = W.prefill_batch("p", [(0, 20), (90, 33)], 24, 8, 128, 16, "bf16", seed=77)
    dev = run_gpu(b)
    kp, vp = oracle_pools(b)
    assert max_err(dev.prefill["out"], oracle.prefill_batch(b, kp, vp)) <= TOL["bf16"]


@pytest.mark.parametrize("src,kv", [("f16", "f16"), ("bf16", "fp8"), ("f16", "fp8")])
def test_prefill_tensor_core_query_dtype_output(src, kv):
    b = W.prefill_batch("p", [(0, 37), (200, 100)], 32, 8, 128, 16, src, kv_dtype=kv, seed=19)
    dev = run_gpu(b, out_dtype="q")
    kp, vp = oracle_pools(b)
    ref = oracle.prefill_batch(b, kp, vp)
    assert rounded_excess(dev.prefill["out"], ref, src, TOL[kv]) <= 0


@pytest.mark.parametrize("src,hq", [("bf16", 64), ("f16", 32)])
def test_prefill_long_chunk_full(src, hq):
    # a 512-row chunk over 4096 tokens of context, Llama-shaped GQA (8 KV heads), every row
    b = W.prefill_batch("p", [(4096, 512)], hq, 8, 128, 16, src, seed=23)
    dev = run_gpu(b)
    kp, vp = oracle_pools(b)
    assert max_err(dev.prefill["out"], oracle.prefill_batch(b, kp, vp)) <= TOL[src]


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_prefill_tensor_core_metadata_errors(kv):
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    b = W.prefill_batch("p", [(40, 70), (10, 5)], 32, 8, 128, 16, "bf16", kv_dtype=kv, seed=31)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.write_step()
    dev.prefill_chunk()
    assert pa.pa_get_device_error() == 0
    dev.prefill["seq_lens"][1] += 1                     # seq_len != q_start + chunk length
    dev.prefill_chunk()
    assert pa.pa_get_device_error() == 4
    dev.prefill["seq_lens"][1] -= 1
    dev.prefill["block_tables"][0, 3] = b.num_blocks + 5  # out-of-range block id
    dev.prefill_chunk()
    assert pa.pa_get_device_error() == 4
    dev.prefill["block_tables"][0, 3] = -2
    dev.prefill_chunk()
    assert pa.pa_get_device_error() == 4


# Batches large enough that the tensor-core kernel puts two 128-row Q tiles in
# each CTA (at least one CTA per SM); the cases above are small enough to use
# one Q tile per CTA.
@pytest.mark.parametrize("src,kv", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "fp8")])
@pytest.mark.parametrize("hq,hkv,chunks", [
    (32, 8, [(100, 300), (7, 300), (640, 257), (0, 299)]),
    (64, 8, [(int(s), 100) for s in range(0, 800, 100)]),
    (8, 8, [(int(s), 256 - s % 7) for s in range(0, 2000, 100)]),
])
@pytest.mark.parametrize("bs", [16, 32])
def test_prefill_two_q_tiles_per_cta(src, kv, hq, hkv, chunks, bs):
    g = hq // hkv
    br = 256 // g
    assert sum(-(-c // br) for _, c in chunks) * hkv >= 152
    b = W.prefill_batch("p", chunks, hq, hkv, 128, bs, src, kv_dtype=kv, seed=hq + len(chunks) + bs)
    dev = run_gpu(b)
    kp, vp = oracle_pools(b)
    ref = oracle.prefill_batch(b, kp, vp)
    assert max_err(dev.prefill["out"], ref) <= TOL[kv]
