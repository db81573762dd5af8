"""Device-side staging of a seeded batch (from ``workloads``) for the CUDA path.

Uploads the batch's host arrays once, allocates the two KV pools filled with
NaN bit patterns, and sequences the batch's setup writes / copies and its step
through the C ABI (``pa_reshape_and_cache``, ``pa_copy_blocks``,
``pa_decode``, ``pa_prefill_chunk``).  It computes nothing itself.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (kv_cache_desc, pa_copy_blocks, pa_decode, pa_decode_workspace_bytes, pa_decode_write, pa_mixed_step,
               pa_prefill_chunk, pa_reshape_and_cache)

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "fp8": torch.uint8}
NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "fp8": 0x7F}


def to_device(bits: np.ndarray, dtype: str, device) -> torch.Tensor:
    """Raw storage bits (uint16 / uint8 numpy) -> device tensor of ``dtype``."""
    if dtype == "fp8":
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).to(device)
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.to(device).view(TORCH_DTYPES[dtype])


def to_bits(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> raw storage bits on the host (uint16 / uint8 numpy)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.uint8:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


class DeviceBatch:
    """A ``workloads.PagedBatch`` resident on one GPU.  ``out_dtype`` "f32"
    keeps the attention outputs in fp32; "q" stores them in the query dtype."""

    def __init__(self, b, device: str | torch.device = "cuda", out_dtype: str = "f32"):
        self.b = b
        self.device = torch.device(device)
        dev = self.device
        shape = (b.num_blocks, b.num_kv_heads, b.block_size, b.head_dim)
        if b.kv_dtype == "fp8":
            self.k_cache = torch.full(shape, NAN_BITS["fp8"], dtype=torch.uint8, device=dev)
        else:
            nan = np.uint16(NAN_BITS[b.kv_dtype]).view(np.int16).item()
            self.k_cache = torch.full(shape, nan, dtype=torch.int16, device=dev).view(TORCH_DTYPES[b.kv_dtype])
        self.v_cache = self.k_cache.clone()
        if np.ndim(b.k_scale) == 0:
            self.head_scales = None
            self.desc = kv_cache_desc(self.k_cache, b.k_scale, b.v_scale)
        else:   # one fp8 scale per KV head
            self.head_scales = (torch.from_numpy(np.ascontiguousarray(b.k_scale, dtype=np.float32)).to(dev),
                                torch.from_numpy(np.ascontiguousarray(b.v_scale, dtype=np.float32)).to(dev))
            self.desc = kv_cache_desc(self.k_cache, 1.0, 1.0, *self.head_scales)
        self.setup_ops = []
        for op in b.setup:
            if hasattr(op, "pairs"):
                self.setup_ops.append(("copy", torch.from_numpy(np.ascontiguousarray(op.pairs)).to(dev)))
            elif len(op.slots):
                self.setup_ops.append(("write", self._write_tensors(op)))
        self.step = self._write_tensors(b.step_write) if b.step_write is not None and len(b.step_write.slots) else None
        self.q = to_device(b.q, b.src_dtype, dev)
        self.block_tables = torch.from_numpy(np.ascontiguousarray(b.block_tables)).to(dev)
        self.seq_lens = torch.from_numpy(np.ascontiguousarray(b.seq_lens)).to(dev)
        odt = torch.float32 if out_dtype == "f32" else self.q.dtype
        self.out = torch.empty(self.q.shape, dtype=odt, device=dev)
        ws = pa_decode_workspace_bytes(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim,
                                       int(b.seq_lens.max()) if b.num_seqs else 0, b.partition_size)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=dev) if ws else None
        self.prefill = None
        if b.prefill is not None:
            p = b.prefill
            self.prefill = dict(
                q=to_device(p.q, b.src_dtype, dev),
                cu_q_lens=torch.from_numpy(p.cu_q_lens).to(dev),
                q_start=torch.from_numpy(p.q_start).to(dev),
                block_tables=torch.from_numpy(np.ascontiguousarray(p.block_tables)).to(dev),
                seq_lens=torch.from_numpy(p.seq_lens).to(dev),
                max_q_len=int(np.diff(p.cu_q_lens).max()) if len(p.q_start) else 0,
                max_seq_len=int(p.seq_lens.max()) if len(p.seq_lens) else 0,
            )
            self.prefill["out"] = torch.empty(self.prefill["q"].shape, dtype=odt, device=dev)

    def _write_tensors(self, op):
        return (to_device(op.k, self.b.src_dtype, self.device), to_device(op.v, self.b.src_dtype, self.device),
                torch.from_numpy(np.ascontiguousarray(op.slots, dtype=np.int64)).to(self.device))

    # ------------------------------------------------------------- the path
    def run_setup(self) -> None:
        for kind, x in self.setup_ops:
            if kind == "copy":
                pa_copy_blocks(self.k_cache, self.v_cache, self.desc, x)
            else:
                pa_reshape_and_cache(x[0], x[1], x[2], self.k_cache, self.v_cache, self.desc)

    def write_step(self) -> None:
        if self.step is not None:
            k, v, s = self.step
            pa_reshape_and_cache(k, v, s, self.k_cache, self.v_cache, self.desc)

    def decode(self) -> torch.Tensor:
        b = self.b
        if b.num_seqs:
            pa_decode(self.q, self.k_cache, self.v_cache, self.desc, self.block_tables, self.seq_lens,
                      int(b.seq_lens.max()), b.scale, self.out, self.workspace, b.partition_size)
        return self.out

    def fused_step_tensors(self, allow_others: bool = False):
        """Per-row new tokens for pa_decode_write: row i's step token is the one
        stored at the slot of its last position (slot -1 and zeros for a row
        without one).  Raises if the step writes anything else, unless
        allow_others (the other tokens are then in self._others)."""
        b = self.b
        if getattr(self, "_fused", None) is None:
            if b.step_write is None:
                raise ValueError("no step write")
            sw = b.step_write
            by_slot = {int(s): t for t, s in enumerate(sw.slots)}
            k = np.zeros((b.num_seqs,) + sw.k.shape[1:], dtype=sw.k.dtype)
            v = np.zeros_like(k)
            slots = np.full(b.num_seqs, -1, dtype=np.int64)
            used = np.zeros(len(sw.slots), dtype=bool)
            for i, L in enumerate(b.seq_lens):
                if L <= 0:
                    continue
                s_last = int(b.block_tables[i][(L - 1) // b.block_size]) * b.block_size + (L - 1) % b.block_size
                t = by_slot.get(s_last)
                if t is None:
                    continue
                k[i], v[i], slots[i] = sw.k[t], sw.v[t], s_last
                used[t] = True
            self._others = None
            if not used.all():
                if not allow_others:
                    raise ValueError("the step writes tokens other than the rows' last positions")
                self._others = self._write_tensors(type(sw)(sw.k[~used], sw.v[~used], sw.slots[~used]))
            self._fused = (to_device(k, b.src_dtype, self.device), to_device(v, b.src_dtype, self.device),
                           torch.from_numpy(slots).to(self.device))
        return self._fused

    def decode_write(self) -> torch.Tensor:
        """The decode step as one call: the step's new tokens written, then attention (pa_decode_write)."""
        b = self.b
        k, v, slots = self.fused_step_tensors()
        if b.num_seqs:
            pa_decode_write(self.q, k, v, slots, self.k_cache, self.v_cache, self.desc, self.block_tables,
                            self.seq_lens, int(b.seq_lens.max()), b.scale, self.out, self.workspace,
                            b.partition_size)
        return self.out

    def prefill_chunk(self) -> torch.Tensor:
        p = self.prefill
        pa_prefill_chunk(p["q"], p["cu_q_lens"], p["q_start"], p["max_q_len"], self.k_cache, self.v_cache, self.desc,
                         p["block_tables"], p["seq_lens"], p["max_seq_len"], self.b.scale, p["out"])
        return p["out"]

    def mixed_step(self, fused: bool = False) -> None:
        """The prefill part and the decode part in one pa_mixed_step call.  fused: the
        chunk's own tokens are written first and the decode rows' new tokens by the
        call itself; else every new token is written first (write_step)."""
        b, p = self.b, self.prefill
        if p is None:
            raise ValueError("the batch has no prefill part")
        new = {}
        if fused:
            k, v, slots = self.fused_step_tensors(allow_others=True)
            if self._others is not None:
                pa_reshape_and_cache(*self._others, self.k_cache, self.v_cache, self.desc)
            new = dict(k_new=k, v_new=v, slot_mapping=slots)
        else:
            self.write_step()
        pa_mixed_step(self.q, self.block_tables, self.seq_lens, int(b.seq_lens.max()) if b.num_seqs else 0, self.out,
                      p["q"], p["cu_q_lens"], p["q_start"], p["max_q_len"], p["block_tables"], p["seq_lens"],
                      p["max_seq_len"], p["out"], self.k_cache, self.v_cache, self.desc, b.scale, self.workspace,
                      b.partition_size, **new)

    def mixed_attention(self) -> None:
        """pa_mixed_step without new tokens: the attention of both parts only."""
        b, p = self.b, self.prefill
        if p is None:
            raise ValueError("the batch has no prefill part")
        pa_mixed_step(self.q, self.block_tables, self.seq_lens, int(b.seq_lens.max()) if b.num_seqs else 0, self.out,
                      p["q"], p["cu_q_lens"], p["q_start"], p["max_q_len"], p["block_tables"], p["seq_lens"],
                      p["max_seq_len"], p["out"], self.k_cache, self.v_cache, self.desc, b.scale, self.workspace,
                      b.partition_size)

    def step_all(self) -> None:
        """One pass of the hot path: write the new tokens, then attend."""
        self.write_step()
        if self.prefill is not None:
            self.prefill_chunk()
        self.decode()
