"""pa_decode_noalloc: paged decode for callers that cannot allocate device memory.

Such callers (code running where cudaMalloc is forbidden or unsafe, or whose
device memory belongs to another framework) get a decode that uses a fixed
scratch array inside the library instead of a caller-provided workspace.
These tests call it through the C ABI and compare it with pa_decode on the
same inputs, twice in a row (the scratch keeps the previous call's contents,
which must not leak into the next result).  Both decode kernels run the same
units in the same order whatever memory holds their workspace, so the
results must equal pa_decode's bit for bit.  The file is named so that
pytest collects it last.
"""
import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    from paged_kv_cache_writes_gb300 import build_lib
    build_lib.build()
    import paged_kv_cache_writes_gb300 as pa
    f = pa.lib().pa_decode_noalloc
    P, I32, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    f.argtypes = [P, ctypes.c_int, I32, I32, P, P, ctypes.POINTER(pa.PaKvCache), P, I32, P, I32, F, I32, P,
                  ctypes.c_int, P]
    f.restype = ctypes.c_int
    return f


def _call(f, dev, out, max_seq_len=None):
    import paged_kv_cache_writes_gb300 as pa
    b = dev.b
    q_code = {"bf16": pa.PA_BF16, "f16": pa.PA_F16}[b.src_dtype]
    return f(dev.q.data_ptr(), q_code, b.num_seqs, b.num_q_heads, dev.k_cache.data_ptr(),
             dev.v_cache.data_ptr(), ctypes.byref(dev.desc), dev.block_tables.data_ptr(),
             dev.block_tables.shape[1], dev.seq_lens.data_ptr(),
             int(b.seq_lens.max()) if max_seq_len is None else max_seq_len, b.scale, b.partition_size,
             out.data_ptr(), pa.PA_F32, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("kernel", ["auto", "cuda_cores"])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_noalloc_equals_pa_decode_on_two_calls(kernel, kv):
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    f = _noalloc_fn()
    # split-KV rows (several partitions), a short row, an empty row
    b = W.decode_batch("noalloc", [3000, 700, 17, 0, 2049, 1], 32, 8, 128, 16, "bf16", kv_dtype=kv, seed=41,
                       partition_size=256)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.write_step()
    with pa.decode_kernel(kernel):
        ref = dev.decode().clone()          # the existing entry point, caller-owned workspace
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        for _ in range(2):
            out = torch.full_like(ref, float("nan"))
            assert _call(f, dev, out) == 0
            torch.cuda.synchronize()
            assert pa.pa_get_device_error() == 0
            assert torch.equal(out.view(torch.int32), ref.view(torch.int32))


def test_noalloc_makes_no_allocation():
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    f = _noalloc_fn()
    b = W.decode_batch("noalloc-mem", [1500, 40, 900], 32, 8, 128, 16, "bf16", seed=43, partition_size=256)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    dev.write_step()
    out = torch.empty_like(dev.out)
    assert _call(f, dev, out) == 0      # first call on the device: set-up (and lazy module loading)
    torch.cuda.synchronize()
    allocs = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call(f, dev, out) == 0
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_rejects_problems_larger_than_its_scratch():
    import paged_kv_cache_writes_gb300 as pa
    from paged_kv_cache_writes_gb300.staging import DeviceBatch
    f = _noalloc_fn()
    b = W.decode_batch("noalloc-big", [40, 50], 32, 8, 128, 16, "bf16", seed=42)
    dev = DeviceBatch(b, "cuda")
    dev.run_setup()
    out = torch.zeros_like(dev.out)
    # a host bound of ~2M tokens needs about 3907 partitions of split-KV partials
    big = 2_000_000
    assert pa.pa_decode_workspace_bytes(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim, big) > (64 << 20)
    assert _call(f, dev, out, max_seq_len=big) == 2          # PA_ERR_UNSUPPORTED, nothing launched
    torch.cuda.synchronize()
    assert float(out.abs().max()) == 0.0
