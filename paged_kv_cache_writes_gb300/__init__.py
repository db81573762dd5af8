"""Python binding of libpa, a PagedAttention hot path for GB300 (sm_103a).

Thin marshalling over the C ABI declared in ``include/pa.h``: every function
here has the name of its C entry point, takes PyTorch CUDA tensors (used only
as device memory), passes their data pointers and the current CUDA stream, and
raises ``PaError`` on a non-OK status.  All arithmetic runs in the library's
CUDA kernels.  There is no CPU fallback: if ``libpa.so`` has not been built,
importing the binding works but every call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

__all__ = [
    "PA_F16", "PA_BF16", "PA_FP8_E4M3", "PA_F32", "PaError", "PaKvCache", "lib", "kv_cache_desc",
    "pa_reshape_and_cache", "pa_copy_blocks", "pa_decode_workspace_bytes", "pa_decode",
    "pa_prefill_chunk", "pa_get_device_error", "pa_status_string", "pa_selftest_wait_timeout",
    "BlockManager", "PaBmStats", "pa_set_decode_kernel", "decode_kernel", "DECODE_KERNELS", "pa_decode_write",
    "pa_mixed_step", "PaDecodePart", "PaPrefillPart",
]

PA_F16, PA_BF16, PA_FP8_E4M3, PA_F32 = 0, 1, 2, 3
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA",
                4: "PA_ERR_DEVICE_CHECK", 5: "PA_ERR_TIMEOUT", 6: "PA_ERR_NO_BLOCKS"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class PaKvCache(ctypes.Structure):
    """Mirror of ``pa_kv_cache``."""
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("k_head_scales", ctypes.c_void_p), ("v_head_scales", ctypes.c_void_p)]


class PaDecodePart(ctypes.Structure):
    """Mirror of ``pa_decode_part``."""
    _fields_ = [("q", ctypes.c_void_p), ("num_seqs", ctypes.c_int32), ("block_tables", ctypes.c_void_p),
                ("max_blocks_per_seq", ctypes.c_int32), ("seq_lens", ctypes.c_void_p),
                ("max_seq_len", ctypes.c_int32), ("partition_size", ctypes.c_int32), ("k_new", ctypes.c_void_p),
                ("v_new", ctypes.c_void_p), ("token_stride", ctypes.c_int64), ("slot_mapping", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t), ("out", ctypes.c_void_p)]


class PaPrefillPart(ctypes.Structure):
    """Mirror of ``pa_prefill_part``."""
    _fields_ = [("q_chunk", ctypes.c_void_p), ("cu_q_lens", ctypes.c_void_p), ("q_start", ctypes.c_void_p),
                ("num_chunks", ctypes.c_int32), ("max_q_len", ctypes.c_int32), ("block_tables", ctypes.c_void_p),
                ("max_blocks_per_seq", ctypes.c_int32), ("seq_lens", ctypes.c_void_p),
                ("max_seq_len", ctypes.c_int32), ("out", ctypes.c_void_p)]


class PaBmStats(ctypes.Structure):
    """Mirror of ``pa_bm_stats``."""
    _fields_ = [("free_blocks", ctypes.c_int32), ("used_blocks", ctypes.c_int32),
                ("shared_blocks", ctypes.c_int32), ("cached_blocks", ctypes.c_int32),
                ("live_sequences", ctypes.c_int32), ("logical_tokens", ctypes.c_int64),
                ("logical_blocks", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpa.so (built by ``build_lib.build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpa.so not built at {LIB_PATH}; run build_lib.build() first")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        L.pa_reshape_and_cache.argtypes = [P, P, ctypes.c_int, I32, I64, P, P, P, ctypes.POINTER(PaKvCache), P]
        L.pa_copy_blocks.argtypes = [P, P, ctypes.POINTER(PaKvCache), P, I32, P]
        L.pa_decode_workspace_bytes.argtypes = [I32, I32, I32, I32, I32, I32]
        L.pa_decode_workspace_bytes.restype = SZ
        L.pa_decode.argtypes = [P, ctypes.c_int, I32, I32, P, P, ctypes.POINTER(PaKvCache), P, I32, P, I32, F,
                                I32, P, SZ, P, ctypes.c_int, P]
        L.pa_decode_write.argtypes = [P, ctypes.c_int, I32, I32, P, P, I64, P, P, P, ctypes.POINTER(PaKvCache), P,
                                      I32, P, I32, F, I32, P, SZ, P, ctypes.c_int, P]
        L.pa_prefill_chunk.argtypes = [P, ctypes.c_int, P, P, I32, I32, I32, P, P, ctypes.POINTER(PaKvCache), P,
                                       I32, P, I32, F, P, ctypes.c_int, P]
        L.pa_mixed_step.argtypes = [ctypes.POINTER(PaDecodePart), ctypes.POINTER(PaPrefillPart), ctypes.c_int, I32,
                                    P, P, ctypes.POINTER(PaKvCache), F, ctypes.c_int, P]
        L.pa_get_device_error.argtypes = [P, ctypes.POINTER(I32)]
        L.pa_set_decode_kernel.argtypes = [I32]
        L.pa_selftest_wait_timeout.argtypes = [P]
        L.pa_status_string.argtypes = [ctypes.c_int]
        L.pa_status_string.restype = ctypes.c_char_p
        VP = ctypes.c_void_p
        L.pa_bm_create.argtypes = [I32, I32, ctypes.c_uint64, ctypes.POINTER(VP)]
        L.pa_bm_destroy.argtypes = [VP]
        L.pa_bm_destroy.restype = None
        L.pa_bm_new_sequence.argtypes = [VP, ctypes.POINTER(I32)]
        L.pa_bm_fork.argtypes = [VP, I32, ctypes.POINTER(I32)]
        L.pa_bm_append.argtypes = [VP, I32, I32, P, P, P, I32, ctypes.POINTER(I32)]
        L.pa_bm_free.argtypes = [VP, I32]
        L.pa_bm_block_table.argtypes = [VP, I32, P, I32, ctypes.POINTER(I32), ctypes.POINTER(I32)]
        L.pa_bm_get_stats.argtypes = [VP, ctypes.POINTER(PaBmStats)]
        for name in ("pa_reshape_and_cache", "pa_copy_blocks", "pa_decode", "pa_prefill_chunk", "pa_set_decode_kernel",
                     "pa_decode_write", "pa_mixed_step",
                     "pa_get_device_error", "pa_selftest_wait_timeout", "pa_bm_create", "pa_bm_new_sequence",
                     "pa_bm_fork", "pa_bm_append", "pa_bm_free", "pa_bm_block_table", "pa_bm_get_stats"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float16:
        return PA_F16
    if t == torch.bfloat16:
        return PA_BF16
    if t in (torch.uint8, torch.float8_e4m3fn):
        return PA_FP8_E4M3
    if t == torch.float32:
        return PA_F32
    raise TypeError(f"unsupported dtype {t}")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor | None, name: str) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _ok(status: int, where: str) -> None:
    if status != 0:
        raise PaError(status, where)


def kv_cache_desc(k_cache: torch.Tensor, k_scale: float = 1.0, v_scale: float = 1.0,
                  k_head_scales: torch.Tensor | None = None, v_head_scales: torch.Tensor | None = None) -> PaKvCache:
    """Descriptor of a pool tensor shaped [num_blocks, num_kv_heads, block_size, head_dim].
    fp8 per-head scales: float32 device tensors [num_kv_heads] (kept alive by the caller)."""
    nb, hkv, bs, d = k_cache.shape
    for t in (k_head_scales, v_head_scales):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (hkv,) or not t.is_contiguous()):
            raise ValueError("per-head scales must be contiguous float32 [num_kv_heads]")
    return PaKvCache(nb, bs, hkv, d, _dtype_code(k_cache.dtype), float(k_scale), float(v_scale),
                     None if k_head_scales is None else k_head_scales.data_ptr(),
                     None if v_head_scales is None else v_head_scales.data_ptr())


def pa_reshape_and_cache(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, cache: PaKvCache, stream=None) -> None:
    """k, v: [T, Hkv, D] (f16/bf16, token stride may exceed Hkv*D); slot_mapping int64 [T]."""
    T = k.shape[0]
    stride = k.stride(0)
    if k.stride()[1:] != (k.shape[2], 1) or v.stride() != k.stride():
        raise ValueError("k and v must be [T, Hkv, D] with unit inner strides and equal strides")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    _ok(lib().pa_reshape_and_cache(k.data_ptr(), v.data_ptr(), _dtype_code(k.dtype), T, stride,
                                   _dev(slot_mapping, "slot_mapping"), _dev(k_cache, "k_cache"),
                                   _dev(v_cache, "v_cache"), ctypes.byref(cache), _stream(stream)),
        "pa_reshape_and_cache")


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, cache: PaKvCache, src_dst_pairs: torch.Tensor,
                   stream=None) -> None:
    """src_dst_pairs: int32 [n, 2] of (src, dst) physical block ids."""
    if src_dst_pairs.dtype != torch.int32:
        raise TypeError("src_dst_pairs must be int32")
    _ok(lib().pa_copy_blocks(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(cache),
                             _dev(src_dst_pairs, "src_dst_pairs"), src_dst_pairs.shape[0], _stream(stream)),
        "pa_copy_blocks")


def pa_decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                              max_seq_len: int, partition_size: int = 0) -> int:
    return int(lib().pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                                               partition_size))


def pa_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, cache: PaKvCache,
              block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, scale: float,
              out: torch.Tensor, workspace: torch.Tensor | None = None, partition_size: int = 0,
              stream=None) -> None:
    """q, out: [B, Hq, D] (out: q's dtype or float32); block_tables int32 [B, max_blocks]; seq_lens int32 [B].
    ``workspace``: uint8 tensor of >= pa_decode_workspace_bytes(...) bytes,
    zero-filled before its first use (None when that size is 0)."""
    B, hq, _ = q.shape
    ws_ptr = _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(lib().pa_decode(_dev(q, "q"), _dtype_code(q.dtype), B, hq, _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                        ctypes.byref(cache), _dev(block_tables, "block_tables"), block_tables.shape[1],
                        _dev(seq_lens, "seq_lens"), int(max_seq_len), float(scale), int(partition_size), ws_ptr,
                        ws_bytes, _dev(out, "out"), _dtype_code(out.dtype), _stream(stream)), "pa_decode")


def pa_decode_write(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                    k_cache: torch.Tensor, v_cache: torch.Tensor, cache: PaKvCache, block_tables: torch.Tensor,
                    seq_lens: torch.Tensor, max_seq_len: int, scale: float, out: torch.Tensor,
                    workspace: torch.Tensor | None = None, partition_size: int = 0, stream=None) -> None:
    """One decode step: row i of k_new / v_new ([B, Hkv, D], q's dtype, unit inner strides) is written at
    slot_mapping[i] (int64 [B]; the slot of position seq_lens[i]-1, or negative), then pa_decode."""
    B, hq, _ = q.shape
    if k_new.stride()[1:] != (k_new.shape[2], 1) or v_new.stride() != k_new.stride():
        raise ValueError("k_new and v_new must be [B, Hkv, D] with unit inner strides and equal strides")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    ws_ptr = _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(lib().pa_decode_write(_dev(q, "q"), _dtype_code(q.dtype), B, hq, _dev(k_new, "k_new"), _dev(v_new, "v_new"),
                              k_new.stride(0), _dev(slot_mapping, "slot_mapping"), _dev(k_cache, "k_cache"),
                              _dev(v_cache, "v_cache"), ctypes.byref(cache), _dev(block_tables, "block_tables"),
                              block_tables.shape[1], _dev(seq_lens, "seq_lens"), int(max_seq_len), float(scale),
                              int(partition_size), ws_ptr, ws_bytes, _dev(out, "out"), _dtype_code(out.dtype),
                              _stream(stream)), "pa_decode_write")


def pa_prefill_chunk(q_chunk: torch.Tensor, cu_q_lens: torch.Tensor, q_start: torch.Tensor, max_q_len: int,
                     k_cache: torch.Tensor, v_cache: torch.Tensor, cache: PaKvCache, block_tables: torch.Tensor,
                     seq_lens: torch.Tensor, max_seq_len: int, scale: float, out: torch.Tensor,
                     stream=None) -> None:
    """q_chunk, out: [total_q, Hq, D] (out: q's dtype or float32); cu_q_lens int32 [n+1]; q_start, seq_lens int32 [n]."""
    _ok(lib().pa_prefill_chunk(_dev(q_chunk, "q_chunk"), _dtype_code(q_chunk.dtype), _dev(cu_q_lens, "cu_q_lens"),
                               _dev(q_start, "q_start"), q_start.shape[0], int(max_q_len), q_chunk.shape[1],
                               _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(cache),
                               _dev(block_tables, "block_tables"), block_tables.shape[1], _dev(seq_lens, "seq_lens"),
                               int(max_seq_len), float(scale), _dev(out, "out"), _dtype_code(out.dtype),
                               _stream(stream)),
        "pa_prefill_chunk")


def pa_mixed_step(q: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                  out: torch.Tensor, q_chunk: torch.Tensor, cu_q_lens: torch.Tensor, q_start: torch.Tensor,
                  max_q_len: int, chunk_block_tables: torch.Tensor, chunk_seq_lens: torch.Tensor,
                  chunk_max_seq_len: int, chunk_out: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                  cache: PaKvCache, scale: float, workspace: torch.Tensor | None = None, partition_size: int = 0,
                  k_new: torch.Tensor | None = None, v_new: torch.Tensor | None = None,
                  slot_mapping: torch.Tensor | None = None, stream=None) -> None:
    """One layer's decode batch (q ... out, with optional new tokens k_new / v_new / slot_mapping as for
    pa_decode_write) and chunked-prefill batch (q_chunk ... chunk_out, as for pa_prefill_chunk) in one call."""
    if (k_new is None) != (v_new is None) or (k_new is None) != (slot_mapping is None):
        raise ValueError("k_new, v_new and slot_mapping go together")
    if slot_mapping is not None and slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    d = PaDecodePart(q=_dev(q, "q"), num_seqs=q.shape[0], block_tables=_dev(block_tables, "block_tables"),
                     max_blocks_per_seq=block_tables.shape[1], seq_lens=_dev(seq_lens, "seq_lens"),
                     max_seq_len=int(max_seq_len), partition_size=int(partition_size),
                     k_new=_dev(k_new, "k_new"), v_new=_dev(v_new, "v_new"),
                     token_stride=0 if k_new is None else k_new.stride(0),
                     slot_mapping=_dev(slot_mapping, "slot_mapping"), workspace=_dev(workspace, "workspace"),
                     workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
                     out=_dev(out, "out"))
    pf = PaPrefillPart(q_chunk=_dev(q_chunk, "q_chunk"), cu_q_lens=_dev(cu_q_lens, "cu_q_lens"),
                       q_start=_dev(q_start, "q_start"), num_chunks=q_start.shape[0], max_q_len=int(max_q_len),
                       block_tables=_dev(chunk_block_tables, "chunk_block_tables"),
                       max_blocks_per_seq=chunk_block_tables.shape[1], seq_lens=_dev(chunk_seq_lens, "chunk_seq_lens"),
                       max_seq_len=int(chunk_max_seq_len), out=_dev(chunk_out, "chunk_out"))
    _ok(lib().pa_mixed_step(ctypes.byref(d), ctypes.byref(pf), _dtype_code(q.dtype), q.shape[1],
                            _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(cache), float(scale),
                            _dtype_code(out.dtype), _stream(stream)), "pa_mixed_step")


def pa_get_device_error(stream=None) -> int:
    """Synchronise the stream, then read and clear the device error word."""
    code = ctypes.c_int32(0)
    _ok(lib().pa_get_device_error(_stream(stream), ctypes.byref(code)), "pa_get_device_error")
    return code.value


def pa_selftest_wait_timeout(stream=None) -> None:
    """Enqueue one warp whose bounded wait expires (records PA_ERR_TIMEOUT, then returns)."""
    _ok(lib().pa_selftest_wait_timeout(_stream(stream)), "pa_selftest_wait_timeout")


DECODE_KERNELS = {"auto": 0, "cuda_cores": 1}


def pa_set_decode_kernel(kernel: str) -> None:
    """Process-wide choice of decode kernel: "auto" (tensor cores where they
    apply) or "cuda_cores"."""
    _ok(lib().pa_set_decode_kernel(DECODE_KERNELS[kernel]), "pa_set_decode_kernel")


@contextlib.contextmanager
def decode_kernel(kernel: str):
    """Use one decode kernel inside the block, then return to "auto"."""
    pa_set_decode_kernel(kernel)
    try:
        yield
    finally:
        pa_set_decode_kernel("auto")


def pa_status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


class BlockManager:
    """Host block manager of one paged pool (``pa_bm_*``): block tables, slots,
    fork with shared blocks, copy-on-write pairs and prefix reuse.  Host only:
    works without a GPU.  Arrays are numpy (int32 tables/ids/pairs, int64 slots)."""

    def __init__(self, num_blocks: int, block_size: int, shuffle_seed: int = 0):
        import numpy as np  # noqa: F401  (numpy arrays are the interface)
        self._h = ctypes.c_void_p()
        self.block_size = int(block_size)
        _ok(lib().pa_bm_create(int(num_blocks), int(block_size), int(shuffle_seed), ctypes.byref(self._h)),
            "pa_bm_create")

    def close(self) -> None:
        if self._h:
            lib().pa_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def new_sequence(self) -> int:
        s = ctypes.c_int32()
        _ok(lib().pa_bm_new_sequence(self._h, ctypes.byref(s)), "pa_bm_new_sequence")
        return s.value

    def fork(self, parent: int) -> int:
        c = ctypes.c_int32()
        _ok(lib().pa_bm_fork(self._h, int(parent), ctypes.byref(c)), "pa_bm_fork")
        return c.value

    def append(self, seq: int, num_tokens: int, token_ids=None):
        """Returns (slots int64[num_tokens], cow pairs int32[k, 2])."""
        import numpy as np
        slots = np.empty(int(num_tokens), dtype=np.int64)
        pairs = np.empty((1, 2), dtype=np.int32)
        ncow = ctypes.c_int32()
        ids = None
        if token_ids is not None:
            ids = np.ascontiguousarray(token_ids, dtype=np.int32)
            if ids.shape != (int(num_tokens),):
                raise ValueError("token_ids must have num_tokens entries")
        _ok(lib().pa_bm_append(self._h, int(seq), int(num_tokens),
                               None if ids is None else ids.ctypes.data, slots.ctypes.data if num_tokens else None,
                               pairs.ctypes.data, 1, ctypes.byref(ncow)), "pa_bm_append")
        return slots, pairs[:ncow.value].copy()

    def free(self, seq: int) -> None:
        _ok(lib().pa_bm_free(self._h, int(seq)), "pa_bm_free")

    def block_table(self, seq: int):
        """Returns (table int32[num_blocks], seq_len)."""
        import numpy as np
        nb, L = ctypes.c_int32(), ctypes.c_int32()
        st = lib().pa_bm_block_table(self._h, int(seq), None, 0, ctypes.byref(nb), ctypes.byref(L))
        if st not in (0, 1):
            _ok(st, "pa_bm_block_table")
        table = np.empty(nb.value, dtype=np.int32)
        _ok(lib().pa_bm_block_table(self._h, int(seq), table.ctypes.data if nb.value else None, nb.value,
                                    ctypes.byref(nb), ctypes.byref(L)), "pa_bm_block_table")
        return table, L.value

    def stats(self) -> PaBmStats:
        st = PaBmStats()
        _ok(lib().pa_bm_get_stats(self._h, ctypes.byref(st)), "pa_bm_get_stats")
        return st
