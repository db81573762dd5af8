"""GPU parity of the cache write and the block copy: bit-exact against the
oracle on the same seeded inputs, with untouched pool bytes left as they were
(the pools start as NaN bit patterns)."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import oracle_pools, run_gpu

pytestmark = pytest.mark.gpu


def _pools_equal(dev, kp, vp):
    from paged_kv_cache_writes_gb300.staging import to_bits
    return np.array_equal(to_bits(dev.k_cache), kp) and np.array_equal(to_bits(dev.v_cache), vp)


@pytest.mark.parametrize("src,kv", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "fp8"), ("f16", "fp8")])
@pytest.mark.parametrize("d,bs", [(128, 16), (64, 32), (128, 32)])
def test_write_bit_exact(src, kv, d, bs):
    b = W.decode_batch("w", [1, 15, 16, 17, 100, 333], 8, 4, d, bs, src, kv_dtype=kv, seed=21)
    dev = run_gpu(b, step=False)
    dev.write_step()
    torch.cuda.synchronize()
    kp, vp = oracle_pools(b)
    assert _pools_equal(dev, kp, vp)


def test_write_skips_negative_slots_and_honours_token_stride():
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import to_bits, to_device
    import oracle
    rng = np.random.default_rng(3)
    T, hkv, d, nb, bs = 40, 2, 64, 16, 16
    fused = W.round_to_bits(rng.standard_normal((T, 3, hkv, d)).astype(np.float32), "bf16")  # q|k|v per token
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[::7] = -1
    dq = to_device(fused, "bf16", "cuda")
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    desc = pa.kv_cache_desc(kc)
    pa.pa_reshape_and_cache(dq[:, 1], dq[:, 2], torch.from_numpy(slots).cuda(), kc, vc, desc)
    torch.cuda.synchronize()
    kp = np.zeros((nb, hkv, bs, d), np.uint16)
    vp = np.zeros_like(kp)
    oracle.reshape_and_cache(np.ascontiguousarray(fused[:, 1]), np.ascontiguousarray(fused[:, 2]), oracle.BF16,
                             slots, kp, vp, oracle.BF16)
    assert np.array_equal(to_bits(kc), kp) and np.array_equal(to_bits(vc), vp)
    assert pa.pa_get_device_error() == 0


def test_write_out_of_range_slot_sets_error_and_writes_nothing():
    import paged_kv_cache_writes_gb300 as pa
    kc = torch.zeros((4, 1, 16, 64), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones((2, 1, 64), dtype=torch.float16, device="cuda")
    slots = torch.tensor([64, 1 << 40], dtype=torch.int64, device="cuda")       # both beyond 4*16
    pa.pa_reshape_and_cache(k, k, slots, kc, vc, pa.kv_cache_desc(kc))
    assert pa.pa_get_device_error() == 4                                          # PA_ERR_DEVICE_CHECK
    assert kc.abs().sum().item() == 0 and vc.abs().sum().item() == 0
    assert pa.pa_get_device_error() == 0                                          # cleared by the read


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_copy_blocks_bit_exact(dtype):
    b = W.shared_prefix_batch(num_prompts=3, prefix_len=64, tail_max=40, num_q_heads=8, num_kv_heads=2, seed=22)
    if dtype == "fp8":
        b.kv_dtype = "fp8"
        b.k_scale = b.v_scale = 0.01
    dev = run_gpu(b, step=True)
    kp, vp = oracle_pools(b)
    assert _pools_equal(dev, kp, vp)


def test_copy_blocks_bad_id_sets_error():
    import paged_kv_cache_writes_gb300 as pa
    kc = torch.arange(4 * 2 * 16 * 64, dtype=torch.int16, device="cuda").view(torch.float16).reshape(4, 2, 16, 64)
    vc = kc.clone()
    before = kc.clone()
    pairs = torch.tensor([[0, 4], [-1, 2]], dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(kc, vc, pa.kv_cache_desc(kc), pairs)
    assert pa.pa_get_device_error() == 4
    assert torch.equal(kc.view(torch.int16), before.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "llama8b", "llama70b", "shared_prefix", "mixed_fp8"])
def test_config_pools_bit_exact(name):
    """Every write and copy of each named workload (setup and step) lands
    bit-exactly where the oracle puts it."""
    b = W.NAMED_WORKLOADS[name]()
    dev = run_gpu(b, step=False)
    dev.write_step()
    torch.cuda.synchronize()
    kp, vp = oracle_pools(b)
    assert _pools_equal(dev, kp, vp)
