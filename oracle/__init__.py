"""fp64 CPU oracle of the PagedAttention hot path (ctypes wrapper of pa_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library (``paged_kv_cache_writes_gb300``) never imports it, and it never
imports the product library: the two share no code.

Every array handed to the oracle is a host numpy array.  16-bit floating point
data (fp16, bf16) is passed as its raw ``uint16`` bit patterns and fp8-e4m3 as
raw ``uint8`` codes, so that the oracle sees exactly the bits the GPU sees.

The arithmetic lives in ``pa_oracle.c``; each function there cites the passage
of the pages it follows.  This module only builds the shared object, marshals
arguments and checks return codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F16, BF16, FP8_E4M3 = 0, 1, 2
DTYPE_CODES = {"f16": F16, "bf16": BF16, "fp8": FP8_E4M3}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_ERRORS = {1: "invalid argument", 2: "index out of range", 3: "out of memory"}


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (fp64, OpenMP, no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        # no OpenMP runtime: the oracle still works, single-threaded
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.or_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.or_f16_to_double.restype = ctypes.c_double
        lib.or_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.or_bf16_to_double.restype = ctypes.c_double
        lib.or_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_to_double.restype = ctypes.c_double
        lib.or_e4m3_encode.argtypes = [ctypes.c_float]
        lib.or_e4m3_encode.restype = ctypes.c_uint8
        lib.or_reshape_and_cache.argtypes = [P, P, I, I64, I64, P, P, P, I64, I, I, I, I, P, P]
        lib.or_reshape_and_cache.restype = I
        lib.or_copy_blocks.argtypes = [P, P, I64, I64, P, I64]
        lib.or_copy_blocks.restype = I
        lib.or_decode.argtypes = [P, I, I, I, P, P, I64, I, I, I, I, P, P, P, I, P, F, P, I, P]
        lib.or_decode.restype = I
        lib.or_prefill.argtypes = [P, I, P, P, I, I, P, P, I64, I, I, I, I, P, P, P, I, F, P]
        lib.or_prefill.restype = I
        lib.or_max_threads.restype = I
        lib.or_set_threads.argtypes = [I]
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: {_ERRORS.get(rc, rc)}")


def _bits_dtype(dt: int):
    return np.uint8 if dt == FP8_E4M3 else np.uint16


# ----------------------------------------------------------------- scalars
def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.or_f16_to_double(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.or_bf16_to_double(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.or_e4m3_to_double(int(c)) for c in flat], dtype=np.float64).reshape(np.shape(codes))


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """fp32 values -> e4m3 codes (RNE, satfinite), one call per element."""
    lib = _load()
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.array([lib.or_e4m3_encode(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(x))


def _scales(x, hkv: int) -> np.ndarray:
    """fp8 scales as one fp32 value per KV head: a per-tensor scale is the same for every head."""
    a = np.asarray(x, dtype=np.float32).reshape(-1)
    if a.size == 1:
        a = np.full(hkv, a[0], dtype=np.float32)
    assert a.shape == (hkv,), "one scale, or one per KV head"
    return np.ascontiguousarray(a)


# -------------------------------------------------------------- cache write
def reshape_and_cache(k: np.ndarray, v: np.ndarray, in_dtype: int, slot_mapping: np.ndarray,
                      k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: int,
                      k_scale=1.0, v_scale=1.0) -> None:
    """Write tokens into the pools in place.  k, v: [T, Hkv, d] bits (token
    stride = Hkv*d); pools: [NB, Hkv, bs, d] bits; slot_mapping int64 [T];
    k_scale / v_scale: one fp8 scale, or one per KV head."""
    lib = _load()
    T, hkv, d = k.shape
    nb, hkv2, bs, d2 = k_cache.shape
    assert (hkv2, d2) == (hkv, d) and v.shape == k.shape and v_cache.shape == k_cache.shape
    assert k.dtype == np.uint16 and k_cache.dtype == _bits_dtype(kv_dtype)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert slots.shape == (T,)
    ks, vs = _scales(k_scale, hkv), _scales(v_scale, hkv)
    _check(lib.or_reshape_and_cache(_ptr(k), _ptr(v), in_dtype, T, hkv * d, _ptr(slots),
                                    _ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d, kv_dtype,
                                    _ptr(ks), _ptr(vs)), "reshape_and_cache")


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs: np.ndarray) -> None:
    """Copy whole physical blocks in place; pairs int32 [n, 2] of (src, dst)."""
    lib = _load()
    pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    nb = k_cache.shape[0]
    block_bytes = k_cache[0].nbytes
    _check(lib.or_copy_blocks(_ptr(k_cache), _ptr(v_cache), nb, block_bytes, _ptr(pairs), len(pairs)),
           "copy_blocks")


# ---------------------------------------------------------------- attention
def decode(q: np.ndarray, q_dtype: int, k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: int,
           block_tables: np.ndarray, seq_lens: np.ndarray, scale: float,
           k_scale=1.0, v_scale=1.0, seq_ids=None) -> np.ndarray:
    """Paged decode in fp64.  q: [B, Hq, d] bits.  Returns float64 [B, Hq, d];
    with ``seq_ids`` only those sequences are evaluated (other rows are NaN)."""
    lib = _load()
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d2 == d
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.full((B, hq, d), np.nan)
    ids = None if seq_ids is None else np.ascontiguousarray(seq_ids, dtype=np.int32)
    ks, vs = _scales(k_scale, hkv), _scales(v_scale, hkv)
    _check(lib.or_decode(_ptr(q), q_dtype, B, hq, _ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d,
                         kv_dtype, _ptr(ks), _ptr(vs), _ptr(bt), bt.shape[1], _ptr(sl),
                         float(scale), _ptr(ids), 0 if ids is None else len(ids), _ptr(out)), "decode")
    return out


def prefill(q: np.ndarray, q_dtype: int, cu_q_lens: np.ndarray, q_start: np.ndarray,
            k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: int, block_tables: np.ndarray,
            scale: float, k_scale=1.0, v_scale=1.0) -> np.ndarray:
    """Chunked prefill in fp64.  q: [total_q, Hq, d] bits.  Returns float64."""
    lib = _load()
    total, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d2 == d
    cu = np.ascontiguousarray(cu_q_lens, dtype=np.int32)
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    assert cu[-1] == total and len(cu) == len(qs) + 1
    out = np.full((total, hq, d), np.nan)
    ks, vs = _scales(k_scale, hkv), _scales(v_scale, hkv)
    _check(lib.or_prefill(_ptr(q), q_dtype, _ptr(cu), _ptr(qs), len(qs), hq, _ptr(k_cache),
                          _ptr(v_cache), nb, bs, hkv, d, kv_dtype, _ptr(ks), _ptr(vs),
                          _ptr(bt), bt.shape[1], float(scale), _ptr(out)), "prefill")
    return out


def max_threads() -> int:
    return _load().or_max_threads()


def set_threads(n: int) -> None:
    _load().or_set_threads(int(n))


def populate(batch, k_pool: np.ndarray, v_pool: np.ndarray, step: bool = True) -> None:
    """Run a batch's setup writes / copies (and, with ``step``, the step's
    new-token write) through the oracle's cache write and block copy, in order."""
    src = DTYPE_CODES[batch.src_dtype]
    kvd = DTYPE_CODES[batch.kv_dtype]
    ops = list(batch.setup) + ([batch.step_write] if step and batch.step_write is not None else [])
    for op in ops:
        if hasattr(op, "pairs"):
            copy_blocks(k_pool, v_pool, op.pairs)
        elif len(op.slots):
            reshape_and_cache(op.k, op.v, src, op.slots, k_pool, v_pool, kvd, batch.k_scale, batch.v_scale)


def decode_batch(batch, k_pool, v_pool, seq_ids=None) -> np.ndarray:
    """Oracle decode of a ``workloads`` batch on pools built by ``populate``."""
    return decode(batch.q, DTYPE_CODES[batch.src_dtype], k_pool, v_pool, DTYPE_CODES[batch.kv_dtype],
                  batch.block_tables, batch.seq_lens, batch.scale, batch.k_scale, batch.v_scale, seq_ids)


def prefill_batch(batch, k_pool, v_pool) -> np.ndarray:
    """Oracle prefill of a batch's prefill part on pools built by ``populate``."""
    p = batch.prefill
    return prefill(p.q, DTYPE_CODES[batch.src_dtype], p.cu_q_lens, p.q_start, k_pool, v_pool,
                   DTYPE_CODES[batch.kv_dtype], p.block_tables, batch.scale, batch.k_scale, batch.v_scale)
