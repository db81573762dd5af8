"""C-ABI checks that need no GPU: the library builds for sm_103a, loads,
exports every entry point the header declares, and rejects bad arguments on
the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_writes_gb300 import build_lib
    build_lib.build()
    import paged_kv_cache_writes_gb300 as pa
    return pa.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:PA_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(pa_[a-z0-9_]+)\s*\(", src, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pa_reshape_and_cache", "pa_decode", "pa_prefill_chunk", "pa_copy_blocks",
                 "pa_decode_workspace_bytes", "pa_get_device_error", "pa_status_string", "pa_decode_write",
                 "pa_mixed_step"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_only_the_c_abi_is_exported(lib):
    """Hidden visibility: the shared object exports the pa_* C symbols and no C++ internals."""
    import subprocess
    from paged_kv_cache_writes_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True).stdout
    syms = [ln.split()[-1] for ln in out.splitlines() if " T " in ln]
    pa_syms = [s for s in syms if s.startswith("pa_")]
    assert sorted(pa_syms) == declared_functions()
    assert not [s for s in syms if s.startswith("_ZN2pa")]


def test_status_strings(lib):
    import paged_kv_cache_writes_gb300 as pa
    assert [pa.pa_status_string(i) for i in range(6)] == [pa.STATUS_NAMES[i] for i in range(6)]
    assert pa.pa_status_string(99) == "PA_ERR_UNKNOWN"


def _desc(**kw):
    import paged_kv_cache_writes_gb300 as pa
    d = dict(num_blocks=64, block_size=16, num_kv_heads=8, head_dim=128, kv_dtype=pa.PA_BF16, k_scale=1.0,
             v_scale=1.0)
    d.update(kw)
    return pa.PaKvCache(**d)


FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced on these paths


def _decode(lib, desc, **kw):
    a = dict(q=FAKE, q_dtype=1, num_seqs=4, num_q_heads=32, k=FAKE, v=FAKE, bt=FAKE, mb=8, sl=FAKE, msl=100,
             scale=0.1, ps=0, ws=None, wsb=0, out=FAKE, odt=1)
    a.update(kw)
    return lib.pa_decode(a["q"], a["q_dtype"], a["num_seqs"], a["num_q_heads"], a["k"], a["v"], ctypes.byref(desc),
                         a["bt"], a["mb"], a["sl"], a["msl"], a["scale"], a["ps"], a["ws"], a["wsb"], a["out"], a["odt"],
                         None)


@pytest.mark.parametrize("kw,desc_kw,want", [
    (dict(num_seqs=0), {}, 0),                                  # zero work: OK, nothing launched
    (dict(num_seqs=-1), {}, 1),
    (dict(num_q_heads=30), {}, 1),                              # Hq % Hkv != 0
    (dict(q=FAKE + 4), {}, 1),                                  # misaligned
    (dict(q=None), {}, 1),
    (dict(out=None), {}, 1),
    (dict(ps=48), {}, 1),                                       # partition not a multiple of 32
    (dict(scale=float("nan")), {}, 1),
    (dict(msl=2000, ws=None), {}, 1),                           # split-KV needs a workspace
    (dict(q_dtype=0), {}, 2),                                   # f16 q with a bf16 cache
    (dict(odt=0), {}, 2),                                       # out must be q dtype or f32
    (dict(odt=2), {}, 2),
    (dict(odt=3, num_seqs=0), {}, 0),                           # f32 out accepted
    ({}, dict(head_dim=96), 2),
    ({}, dict(block_size=8), 2),
    ({}, dict(kv_dtype=7), 2),
    ({}, dict(kv_dtype=2, k_scale=0.0), 1),                     # fp8 needs a positive scale
    ({}, dict(num_blocks=0), 1),
    ({}, dict(num_blocks=1 << 30), 2),                          # rows beyond int32 TMA coordinates
])
def test_decode_host_validation(lib, kw, desc_kw, want):
    assert _decode(lib, _desc(**desc_kw), **kw) == want


def test_reshape_and_cache_validation(lib):
    d = _desc()
    f = lib.pa_reshape_and_cache
    assert f(FAKE, FAKE, 1, 0, 1024, FAKE, FAKE, FAKE, ctypes.byref(d), None) == 0
    assert f(FAKE, FAKE, 1, -1, 1024, FAKE, FAKE, FAKE, ctypes.byref(d), None) == 1
    assert f(FAKE, FAKE, 1, 4, 1000, FAKE, FAKE, FAKE, ctypes.byref(d), None) == 1      # stride < Hkv*D
    assert f(FAKE, FAKE, 1, 4, 1028, FAKE, FAKE, FAKE, ctypes.byref(d), None) == 1      # stride % 8
    assert f(FAKE, FAKE, 0, 4, 1024, FAKE, FAKE, FAKE, ctypes.byref(d), None) == 2      # f16 into bf16 cache
    assert f(FAKE, FAKE, 2, 4, 1024, FAKE, FAKE, FAKE, ctypes.byref(d), None) == 2      # fp8 input
    assert f(FAKE, FAKE, 1, 4, 1024, FAKE + 4, FAKE, FAKE, ctypes.byref(d), None) == 1  # slots misaligned
    assert f(FAKE, FAKE, 1, 4, 1024, FAKE, None, FAKE, ctypes.byref(d), None) == 1
    assert f(FAKE, FAKE, 1, 4, 1024, FAKE, FAKE, FAKE, None, None) == 1


def test_copy_blocks_validation(lib):
    d = _desc()
    f = lib.pa_copy_blocks
    assert f(FAKE, FAKE, ctypes.byref(d), FAKE, 0, None) == 0
    assert f(FAKE, FAKE, ctypes.byref(d), FAKE, -2, None) == 1
    assert f(FAKE, FAKE, ctypes.byref(d), None, 3, None) == 1
    assert f(None, FAKE, ctypes.byref(d), FAKE, 3, None) == 1


def test_prefill_validation(lib):
    d = _desc()
    f = lib.pa_prefill_chunk
    ok = (FAKE, 1, FAKE, FAKE, 1, 64, 32, FAKE, FAKE, ctypes.byref(d), FAKE, 8, FAKE, 128, 0.1, FAKE, 3, None)
    assert f(*ok[:4], 0, *ok[5:]) == 0                      # no chunks
    assert f(*ok[:5], 0, *ok[6:]) == 0                      # empty chunks
    assert f(*ok[:4], -1, *ok[5:]) == 1
    assert f(*ok[:6], 31, *ok[7:]) == 1                     # Hq % Hkv
    assert f(ok[0], 0, *ok[2:]) == 2                        # f16 q, bf16 cache
    assert f(*ok[:2], None, *ok[3:]) == 1
    assert f(*ok[:16], 2, None) == 2                        # fp8 output


def test_workspace_size(lib):
    import paged_kv_cache_writes_gb300 as pa
    hdr, cnt = 256, 256 * 64 * 4
    # one partition: header, item list and counters only
    assert pa.pa_decode_workspace_bytes(256, 64, 8, 128, 512, 0) == hdr + 256 * 4 + cnt
    n = pa.pa_decode_workspace_bytes(256, 64, 8, 128, 8192, 512)
    parts = 16
    items = 256 * parts * 4
    acc = 256 * 64 * parts * 128 * 4
    ml = 256 * 64 * parts * 8
    jobs = 256 * 64 * 16                                                      # merge list (split rows)
    assert n == hdr + items + acc + ml + cnt + jobs                           # all multiples of 256
    assert pa.pa_decode_workspace_bytes(256, 64, 8, 128, 8192, 2048) == n     # partitions above 512 act as 512
    assert pa.pa_decode_workspace_bytes(4, 30, 8, 128, 8192, 0) == 0         # invalid -> 0
    assert pa.pa_decode_workspace_bytes(4, 32, 8, 128, 8192, 48) == 0


def test_per_head_scale_validation(lib):
    import paged_kv_cache_writes_gb300 as pa
    f = lib.pa_reshape_and_cache
    # per-head scales with a 16-bit cache, or only one of the two arrays, or misaligned
    for d in (_desc(k_head_scales=FAKE, v_head_scales=FAKE),
              _desc(kv_dtype=pa.PA_FP8_E4M3, k_head_scales=FAKE),
              _desc(kv_dtype=pa.PA_FP8_E4M3, k_head_scales=FAKE + 2, v_head_scales=FAKE)):
        assert f(FAKE, FAKE, 1, 4, 1024, FAKE, FAKE, FAKE, ctypes.byref(d), None) == 1
    ok = _desc(kv_dtype=pa.PA_FP8_E4M3, k_head_scales=FAKE, v_head_scales=FAKE)
    assert f(FAKE, FAKE, 1, 0, 1024, FAKE, FAKE, FAKE, ctypes.byref(ok), None) == 0      # valid, no tokens


def test_mixed_step_validation(lib):
    """pa_mixed_step checks both parts before it launches anything."""
    import paged_kv_cache_writes_gb300 as pa
    d = _desc()

    def parts(**kw):
        dp = dict(q=FAKE, num_seqs=4, block_tables=FAKE, max_blocks_per_seq=8, seq_lens=FAKE, max_seq_len=100,
                  partition_size=0, k_new=None, v_new=None, token_stride=0, slot_mapping=None, workspace=None,
                  workspace_bytes=0, out=FAKE)
        pp = dict(q_chunk=FAKE, cu_q_lens=FAKE, q_start=FAKE, num_chunks=1, max_q_len=64, block_tables=FAKE,
                  max_blocks_per_seq=8, seq_lens=FAKE, max_seq_len=128, out=FAKE)
        for k, v in kw.items():
            (dp if k.startswith("d_") else pp)[k[2:]] = v
        return pa.PaDecodePart(**dp), pa.PaPrefillPart(**pp)

    def call(q_dtype=1, hq=32, odt=1, **kw):
        dp, pp = parts(**kw)
        return lib.pa_mixed_step(ctypes.byref(dp), ctypes.byref(pp), q_dtype, hq, FAKE, FAKE, ctypes.byref(d), 0.1,
                                 odt, None)

    dp, pp = parts()
    assert lib.pa_mixed_step(None, ctypes.byref(pp), 1, 32, FAKE, FAKE, ctypes.byref(d), 0.1, 1, None) == 1
    assert lib.pa_mixed_step(ctypes.byref(dp), None, 1, 32, FAKE, FAKE, ctypes.byref(d), 0.1, 1, None) == 1
    assert lib.pa_mixed_step(ctypes.byref(dp), ctypes.byref(pp), 1, 32, FAKE, FAKE, None, 0.1, 1, None) == 1
    assert call(d_num_seqs=0, p_num_chunks=0) == 0           # nothing to do
    assert call(p_num_chunks=-1) == 1                        # prefill part invalid
    assert call(p_cu_q_lens=None) == 1
    assert call(hq=31) == 1                                  # Hq % Hkv
    assert call(q_dtype=0) == 2                              # f16 q, bf16 cache
    assert call(odt=2) == 2                                  # fp8 output
    assert call(d_num_seqs=-1) == 1                          # decode part invalid
    assert call(d_k_new=FAKE) == 1                           # new tokens: all three or none
    assert call(d_k_new=FAKE, d_v_new=FAKE, d_slot_mapping=FAKE, d_token_stride=7) == 1
    assert call(d_workspace=None) == 1                       # decode workspace missing
