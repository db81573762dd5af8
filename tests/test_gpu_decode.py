"""GPU parity of paged decode against the fp64 oracle, element by element.

Two kernels serve pa_decode: the tensor-core one (chosen by default for
head_dim 128 with 1..16 query heads per KV head and head_dim 64 with 1..8,
a group running padded to 4, 8 or 16 rows; one head per KV head only with
an fp8 cache) and the CUDA-core one (every other shape, or every shape once
selected with pa_set_decode_kernel); both are checked here.

Tolerance (max abs error): 2e-3 for f16/bf16 caches, 2e-2 for an fp8-e4m3
cache (the oracle dequantises the same codes with the same scales).  Shapes
span several tiles and partitions with ragged tails; the named workloads run
at full size and every output element is compared with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_writes_gb300 as pa
import workloads as W
from _gpu import TOL, max_err, oracle_pools, rounded_excess, run_gpu

pytestmark = pytest.mark.gpu

EDGE_LENS = [1, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1000, 1537]


def _check(b, seq_ids=None):
    dev = run_gpu(b)
    kp, vp = oracle_pools(b)
    ref = oracle.decode_batch(b, kp, vp, seq_ids=seq_ids)
    got = dev.out if seq_ids is None else dev.out[torch.as_tensor(seq_ids, device=dev.out.device).long()]
    ref = ref if seq_ids is None else ref[np.asarray(seq_ids)]
    err = max_err(got, ref)
    assert err <= TOL[b.kv_dtype], err
    return dev, err


def test_tiny_config():
    _check(W.cfg_tiny())


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (16, 2), (32, 8), (64, 8), (12, 4), (6, 2), (5, 5), (40, 8),
                                    (96, 8), (16, 8)])
@pytest.mark.parametrize("d,bs", [(128, 16), (64, 32), (128, 32), (64, 16)])
def test_shapes_bf16(hq, hkv, d, bs):
    _check(W.decode_batch("s", EDGE_LENS, hq, hkv, d, bs, "bf16", seed=hq * 7 + d + bs, partition_size=512))


@pytest.mark.parametrize("kv,src", [("f16", "f16"), ("fp8", "bf16"), ("fp8", "f16")])
@pytest.mark.parametrize("hq,hkv,d,bs", [(32, 8, 128, 16), (64, 8, 128, 32), (8, 8, 64, 16), (16, 4, 64, 32),
                                         (64, 8, 64, 16), (24, 8, 128, 16), (40, 8, 128, 32), (8, 8, 128, 16)])
def test_shapes_other_dtypes(kv, src, hq, hkv, d, bs):
    _check(W.decode_batch("s", EDGE_LENS, hq, hkv, d, bs, src, kv_dtype=kv, seed=hq + d + bs, partition_size=512))


@pytest.mark.parametrize("kv,src", [("f16", "f16"), ("fp8", "bf16"), ("fp8", "f16")])
@pytest.mark.parametrize("hq,hkv,d", [(24, 2, 128), (13, 1, 128), (10, 2, 64), (14, 2, 64)])
def test_padded_groups_other_dtypes(kv, src, hq, hkv, d):
    # groups of 12, 13, 5 and 7 query heads per KV head: run padded to 16 or 8 rows
    _check(W.decode_batch("pad", EDGE_LENS, hq, hkv, d, 16, src, kv_dtype=kv, seed=hq + hkv + d, partition_size=512))


@pytest.mark.parametrize("kv,src", [("bf16", "bf16"), ("f16", "f16"), ("fp8", "bf16"), ("fp8", "f16")])
@pytest.mark.parametrize("hq,hkv,bs", [(32, 2, 16), (64, 4, 32), (16, 1, 16)])
def test_sixteen_heads_per_kv_head(kv, src, hq, hkv, bs):
    _check(W.decode_batch("g16", EDGE_LENS, hq, hkv, 128, bs, src, kv_dtype=kv, seed=hq + hkv + bs,
                          partition_size=512))


@pytest.mark.parametrize("kv,src", [("bf16", "bf16"), ("f16", "f16"), ("fp8", "bf16")])
@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 16), (64, 8, 32), (16, 2, 16), (32, 2, 32)])
def test_cuda_core_kernel_on_tensor_core_shapes(kv, src, hq, hkv, bs):
    """The shapes the tensor-core kernel takes by default, through the CUDA-core kernel."""
    b = W.decode_batch("cc", EDGE_LENS, hq, hkv, 128, bs, src, kv_dtype=kv, seed=hq * 3 + hkv + bs,
                       partition_size=512)
    with pa.decode_kernel("cuda_cores"):
        _check(b)


def test_both_kernels_agree_on_the_llama70b_shape():
    b = W.decode_batch("both", [1, 129, 512, 513, 1000, 2047, 4100, 8192], 64, 8, 128, 16, "bf16", seed=41)
    tc = run_gpu(b).out.clone()
    with pa.decode_kernel("cuda_cores"):
        cc = run_gpu(b).out.clone()
    kp, vp = oracle_pools(b)
    ref = oracle.decode_batch(b, kp, vp)
    assert max_err(tc, ref) <= TOL["bf16"] and max_err(cc, ref) <= TOL["bf16"]
    assert (tc - cc).abs().max().item() <= 2 * TOL["bf16"]


@pytest.mark.parametrize("ps", [0, 32, 96, 512, 2048])
def test_partition_sizes_agree(ps):
    b = W.decode_batch("p", [1, 40, 700, 2049, 3000], 16, 2, 128, 16, "bf16", seed=31, partition_size=ps)
    _check(b)


def test_single_token_context_returns_v_exactly():
    b = W.decode_batch("one", [1] * 9, 16, 4, 128, 32, "bf16", seed=32)
    dev = run_gpu(b, out_dtype="q")
    v = torch.from_numpy(b.step_write.v.view(np.int16)).cuda().view(torch.bfloat16)   # [B, Hkv, D]
    want = v.repeat_interleave(4, dim=1)
    assert torch.equal(dev.out.view(torch.int16), want.contiguous().view(torch.int16))


@pytest.mark.parametrize("src,kv", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "fp8")])
def test_query_dtype_outputs(src, kv):
    """Outputs stored in the query dtype: within the tolerance plus half an
    ulp of the stored value (the round-to-nearest-even storage step)."""
    b = W.decode_batch("q", EDGE_LENS, 32, 8, 128, 16, src, kv_dtype=kv, seed=36, partition_size=512)
    dev = run_gpu(b, out_dtype="q")
    assert dev.out.dtype != torch.float32
    kp, vp = oracle_pools(b)
    ref = oracle.decode_batch(b, kp, vp)
    assert rounded_excess(dev.out, ref, src, TOL[kv]) <= 0


def test_zero_length_sequences():
    b = W.decode_batch("z", [0, 5, 0, 600], 8, 2, 64, 16, "bf16", seed=33, partition_size=256)
    dev, _ = _check(b)
    assert dev.out[0].abs().max().item() == 0 and dev.out[2].abs().max().item() == 0


def test_workspace_contents_ignored_and_reusable():
    """Each call rebuilds its workspace: garbage left in it changes nothing,
    and repeated calls give bit-identical outputs."""
    b = W.decode_batch("r", [3000, 100, 2500, 0, 17], 16, 2, 128, 16, "bf16", seed=34, partition_size=256)
    dev = run_gpu(b)
    first = dev.out.clone()
    for fill in (0xFF, 0x00, 0x5A):
        dev.workspace.fill_(fill)
        dev.decode()
        torch.cuda.synchronize()
        assert torch.equal(dev.out.view(torch.int32), first.view(torch.int32))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_back_to_back_calls_share_one_workspace(kv):
    """Calls on one stream, with no synchronisation between them, may share a
    workspace: each call's plan kernel waits for the stream's previous decode
    before rebuilding the work list (it is launched as a programmatic
    dependent, so it starts while that decode finishes).  Two different
    batches, alternated three times, each checked against the oracle."""
    a = W.decode_batch("bb-a", [3000, 100, 2500, 0, 17, 4100, 777], 64, 8, 128, 32, "bf16", kv_dtype=kv, seed=61,
                       partition_size=512)
    c = W.decode_batch("bb-c", [64, 5000, 1, 2049, 900], 64, 8, 128, 32, "bf16", kv_dtype=kv, seed=62,
                       partition_size=512)
    da, dc = run_gpu(a), run_gpu(c)
    shared = torch.zeros(max(da.workspace.numel(), dc.workspace.numel()), dtype=da.workspace.dtype,
                         device=da.workspace.device)
    da.workspace = shared[: da.workspace.numel()]
    dc.workspace = shared[: dc.workspace.numel()]
    for d in (da, dc):
        d.out.fill_(float("nan"))
    for _ in range(3):
        da.decode()
        dc.decode()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    for b, d in ((a, da), (c, dc)):
        kp, vp = oracle_pools(b)
        ref = oracle.decode_batch(b, kp, vp)
        assert max_err(d.out, ref) <= TOL[kv]


@pytest.mark.parametrize("kv", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8), (128, 16)])
def test_head_dim_64_batch_both_kernels(kv, hq, hkv):
    # a bandwidth-sized head_dim-64 batch (128 sequences of 512..4096 tokens): the tensor-core
    # kernel against the oracle in full, and against the CUDA-core kernel
    lens = np.random.default_rng(101).integers(512, 4097, size=128)
    b = W.decode_batch("d64", lens, hq, hkv, 64, 16, kv, seed=5, partition_size=512)
    tc, _ = _check(b)
    tc_out = tc.out.clone()
    with pa.decode_kernel("cuda_cores"):
        cc, _ = _check(b)
    assert (tc_out - cc.out).abs().max().item() <= 2 * TOL[kv]


@pytest.mark.parametrize("q", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8), (128, 16)])
def test_head_dim_64_fp8_batch_both_kernels(q, hq, hkv):
    # the same batch with an e4m3 cache (64-byte rows, 64-byte swizzle on the tensor-core path)
    lens = np.random.default_rng(102).integers(512, 4097, size=128)
    b = W.decode_batch("d64 fp8", lens, hq, hkv, 64, 16, q, kv_dtype="fp8", seed=6, partition_size=512)
    tc, _ = _check(b)
    tc_out = tc.out.clone()
    with pa.decode_kernel("cuda_cores"):
        cc, _ = _check(b)
    assert (tc_out - cc.out).abs().max().item() <= 2 * TOL["fp8"]


@pytest.mark.parametrize("hq", [24, 40])
def test_gqa_layer_full(hq):
    # the benchmark's decode layers with 3 and 5 query heads per KV head: every row and element
    _check(W.cfg_gqa(hq))


@pytest.mark.parametrize("hq", [32, 64])
def test_head_dim_64_layer_full(hq):
    # the benchmark's head_dim-64 decode layers (256 sequences): every row and element
    _check(W.cfg_d64(num_q_heads=hq))


def test_llama8b_full():
    _check(W.cfg_llama8b())


def test_llama70b_full():
    # the benchmark workload: all 256 sequences, every head and element
    _check(W.cfg_llama70b())


def test_llama70b_full_cuda_core_kernel():
    with pa.decode_kernel("cuda_cores"):
        _check(W.cfg_llama70b())


def test_shared_prefix_full():
    b = W.cfg_shared_prefix()
    _check(b)


@pytest.mark.parametrize("cfg,scales", [("llama8b", "tensor"), ("llama70b", "tensor"), ("llama70b", "head")])
def test_decode_shapes_with_fp8_cache_full(cfg, scales):
    # the decode-only workloads with the cache stored as e4m3 (same values; per-tensor or per-head scales)
    b = {"llama8b": W.cfg_llama8b, "llama70b": W.cfg_llama70b}[cfg](kv_dtype="fp8", fp8_scales=scales)
    assert b.kv_dtype == "fp8"
    _check(b)


def test_mixed_fp8_decode_part_full():
    _check(W.cfg_mixed_fp8())


@pytest.mark.parametrize("kernel", ["auto", "cuda_cores"])
def test_bad_block_id_sets_error_without_fault(kernel):
    b = W.decode_batch("bad", [40, 70], 8, 2, 128, 16, "bf16", seed=35)
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.write_step()
    with pa.decode_kernel(kernel):
        dev.block_tables[1, 2] = b.num_blocks + 5        # out of range
        dev.decode()
        assert pa.pa_get_device_error() == 4
        dev.block_tables[1, 2] = -3
        dev.decode()
        assert pa.pa_get_device_error() == 4
