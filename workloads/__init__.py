"""Seeded synthetic inputs for the PagedAttention hot path.

This module is shared by the oracle side and the CUDA side of every test and of
the benchmark.  It holds none of the method's arithmetic: no attention, no
softmax, no fp8 encoding.  What it does is what a serving engine's host-side
block manager does before a kernel runs:

* draw sequence lengths and N(0,1) query/key/value values (rounded to the
  16-bit storage type, ties to even);
* hand out physical blocks from a seeded permutation of the pool and build the
  per-sequence block tables ("Inside vLLM Architecture", section "The Block
  Table Mapping Subsystem": blocks come from a free list, the table maps a
  sequence's logical block to a physical block);
* turn each token position into a cache slot, ``block_table[p // bs] * bs +
  p % bs`` -- the slot arithmetic of ``allocate_slot`` in that same section;
* for shared-prefix sampling, point the branches of one prompt at the same
  physical prefix blocks and list the copy-on-write (src, dst) block pairs
  ("High-Throughput LLM Serving with vLLM & PagedAttention", section
  "2. Virtual Memory Paging Applied to GPUs").

Each side builds its own KV pool from these inputs through its own cache write,
starting from a pool filled with NaN bit patterns, so that any read of a slot
that was never written shows up as NaN.  Block-table padding entries point at
a spare physical block that is never written (all NaN).

The five named workloads follow the configurations these tests and the
benchmark are quoted on (Llama-3-8B / 70B shaped GQA layers, shared-prefix
sampling, chunked prefill with an fp8 KV cache); see ``NAMED_WORKLOADS``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "fp8": 0x7F}


def round_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> raw 16-bit storage bits, round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32)
        r = u >> 16
        r &= 1
        r += 0x7FFF
        r += u            # finite inputs only: no carry out of 32 bits below NaN
        r >>= 16
        return r.astype(np.uint16)
    raise ValueError(dtype)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Raw 16-bit storage bits -> float32 (exact)."""
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


_CHUNK = 1 << 22


def _normal_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0,1) samples rounded to ``dtype`` bits.  One 64-bit key is drawn from
    ``rng``; chunk c of the output comes from default_rng([key, c]), so the
    result does not depend on how many threads fill the chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    key = int(rng.integers(0, 2**63))

    def fill(c):
        s, e = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.default_rng([key, c])
        out[s:e] = round_to_bits(g.standard_normal(e - s, dtype=np.float32), dtype)

    nchunks = -(-n // _CHUNK)
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


@dataclass
class WriteOp:
    """Tokens to scatter into the cache: k, v [T, Hkv, d] bits, slots int64 [T]."""
    k: np.ndarray
    v: np.ndarray
    slots: np.ndarray


@dataclass
class CopyOp:
    """Copy-on-write block pairs, int32 [n, 2] of (src, dst)."""
    pairs: np.ndarray


@dataclass
class PrefillPart:
    """Query chunks over paged context; sequences in their own table rows."""
    q: np.ndarray            # [total_q, Hq, d] bits (src dtype)
    cu_q_lens: np.ndarray    # int32 [n+1]
    q_start: np.ndarray      # int32 [n]
    block_tables: np.ndarray  # int32 [n, max_blocks]
    seq_lens: np.ndarray     # int32 [n] = q_start + chunk length


@dataclass
class PagedBatch:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    src_dtype: str           # dtype of q and of K/V before caching: "f16" | "bf16"
    kv_dtype: str            # cache dtype: src_dtype or "fp8"
    num_blocks: int
    pad_block: int           # spare physical block, never written
    block_tables: np.ndarray  # int32 [B, max_blocks] (decode sequences)
    seq_lens: np.ndarray     # int32 [B], includes the token decoded this step
    q: np.ndarray            # [B, Hq, d] bits
    scale: float             # softmax scale (a float32 value)
    setup: list = field(default_factory=list)   # WriteOp / CopyOp run before the step
    step_write: WriteOp | None = None           # new tokens written inside the step
    prefill: PrefillPart | None = None
    k_scale: float | np.ndarray = 1.0   # fp8: one scale, or fp32 [Hkv] (one per KV head)
    v_scale: float | np.ndarray = 1.0
    partition_size: int = 0  # 0 = let the library choose
    blocks_unshared: int = 0  # physical blocks the same batch needs without sharing

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_seq_len(self) -> int:
        m = int(self.seq_lens.max()) if self.num_seqs else 0
        if self.prefill is not None and len(self.prefill.seq_lens):
            m = max(m, int(self.prefill.seq_lens.max()))
        return m

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "fp8" else 2

    def decode_kv_bytes(self) -> int:
        """Algorithmic K+V bytes one decode pass reads: each context token's K
        and V row once per KV head (the GQA group shares the read)."""
        return int(self.seq_lens.astype(np.int64).sum()) * 2 * self.num_kv_heads * self.head_dim * self.kv_elem_bytes

    def blocks_used(self) -> int:
        ids = set(np.unique(self.block_tables).tolist())
        if self.prefill is not None:
            ids |= set(np.unique(self.prefill.block_tables).tolist())
        ids.discard(self.pad_block)
        return len(ids)


class _Pool:
    """Seeded free list: physical block ids handed out in a permuted order."""

    def __init__(self, rng: np.random.Generator, num_blocks: int):
        self.order = rng.permutation(num_blocks).astype(np.int64)
        self.pad = int(self.order[-1])       # never handed out
        self.next = 0
        self.limit = num_blocks - 1

    def take(self, n: int) -> np.ndarray:
        if self.next + n > self.limit:
            raise ValueError("pool too small")
        out = self.order[self.next:self.next + n]
        self.next += n
        return out


def _pool_size(needed: int, factor: int = 2, round_to: int = 1024) -> int:
    return max(round_to, -(-(factor * needed + 1) // round_to) * round_to)


def slots_for(table_row: np.ndarray, positions: np.ndarray, bs: int) -> np.ndarray:
    """Cache slot of each token position (allocate_slot's addressing)."""
    positions = np.asarray(positions, dtype=np.int64)
    return table_row[positions // bs].astype(np.int64) * bs + positions % bs


def _tables(rows: list, pad: int) -> np.ndarray:
    mb = max(1, max((len(r) for r in rows), default=1))
    bt = np.full((len(rows), mb), pad, dtype=np.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = r
    return bt


def decode_batch(name: str, lens, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                 src_dtype: str, kv_dtype: str | None = None, seed: int = 0, layout_seed: int | None = None,
                 num_blocks: int | None = None, partition_size: int = 0,
                 scale: float | None = None, fp8_scales: str = "tensor") -> PagedBatch:
    """A decode batch: sequence i has ``lens[i]`` tokens, the last of which is
    the new token written inside the step; the others are existing context.

    ``seed`` draws the values, ``layout_seed`` (default: seed) the physical
    placement, so that one logical batch can be laid out several ways."""
    kv_dtype = kv_dtype or src_dtype
    lens = np.asarray(lens, dtype=np.int64)
    B, bs = len(lens), block_size
    vrng = np.random.default_rng(seed)
    lrng = np.random.default_rng(seed if layout_seed is None else layout_seed)
    nblk = -(-lens // bs)
    needed = int(nblk.sum())
    nb = num_blocks if num_blocks is not None else _pool_size(needed)
    pool = _Pool(lrng, nb)
    rows = [pool.take(int(n)) for n in nblk]
    bt = _tables(rows, pool.pad)
    # values: q, then all tokens of all sequences in sequence order
    q = _normal_bits(vrng, (B, num_q_heads, head_dim), src_dtype)
    T = int(lens.sum())
    k_all = _normal_bits(vrng, (T, num_kv_heads, head_dim), src_dtype)
    v_all = _normal_bits(vrng, (T, num_kv_heads, head_dim), src_dtype)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    slots = np.concatenate([slots_for(bt[i], np.arange(lens[i]), bs) for i in range(B)]) if T else \
        np.zeros(0, np.int64)
    is_new = np.zeros(T, dtype=bool)
    is_new[(starts + lens - 1)[lens > 0]] = True
    ctx = WriteOp(k_all[~is_new], v_all[~is_new], slots[~is_new])
    new = WriteOp(k_all[is_new], v_all[is_new], slots[is_new])
    ks, vs = _fp8_scales([k_all], [v_all], src_dtype, fp8_scales == "head") if kv_dtype == "fp8" else (1.0, 1.0)
    return PagedBatch(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      block_size=bs, src_dtype=src_dtype, kv_dtype=kv_dtype, num_blocks=nb, pad_block=pool.pad,
                      block_tables=bt, seq_lens=lens.astype(np.int32), q=q,
                      scale=float(np.float32(1.0) / np.sqrt(np.float32(head_dim))) if scale is None else scale,
                      setup=[ctx], step_write=new, k_scale=ks, v_scale=vs, partition_size=partition_size,
                      blocks_unshared=needed)


def _amax(bits: np.ndarray, src_dtype: str) -> np.float32:
    """max |x| of finite 16-bit floats: the magnitude bits order like the values."""
    m = np.uint16(0)
    flat = bits.reshape(-1)
    for s in range(0, flat.size, 1 << 26):
        part = flat[s:s + (1 << 26)] & np.uint16(0x7FFF)
        m = max(m, part.max(initial=0))
    return bits_to_f32(np.array([m], np.uint16), src_dtype)[0]


def _fp8_scales(k_parts, v_parts, src_dtype: str, per_head: bool = False):
    """Scales amax(|x|) / 448 in fp32 (448 = largest E4M3 magnitude), the amax
    taken over every token of the tensor (given as a list of [..., Hkv, d]
    parts): one per tensor, or with ``per_head`` one per KV head (fp32 array)."""
    def one(parts):
        amax = max(_amax(p, src_dtype) for p in parts)
        return float(np.float32(amax) / np.float32(448.0)) if amax > 0 else 1.0
    def heads(parts):
        hkv = parts[0].shape[-2]
        return np.array([one([p[..., h, :] for p in parts]) for h in range(hkv)], dtype=np.float32)
    if per_head:
        return heads(k_parts), heads(v_parts)
    return one(k_parts), one(v_parts)


def shared_prefix_batch(name: str = "shared-prefix sampling", num_prompts: int = 32, branches: int = 4,
                        prefix_len: int = 2048, tail_max: int = 256, num_q_heads: int = 32,
                        num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16,
                        src_dtype: str = "bf16", seed: int = 3, shared: bool = True) -> PagedBatch:
    """Parallel sampling: ``branches`` continuations of each prompt.  With
    ``shared`` the branches point at the prompt's physical prefix blocks; the
    last prefix block is copy-on-written for branches 1.. before the tails are
    written.  Without ``shared`` every branch holds a private copy of the
    prefix (same values), the unshared layout the saving is measured against."""
    bs = block_size
    vrng = np.random.default_rng(seed)
    lrng = np.random.default_rng(seed + 1000)
    tails = vrng.integers(0, tail_max + 1, size=(num_prompts, branches))
    lens = (prefix_len + tails + 1).astype(np.int64)            # +1: token decoded this step
    pblk = -(-prefix_len // bs)
    nblk = -(-lens // bs)
    unshared_need = int(nblk.sum())
    nb = _pool_size(unshared_need)
    pool = _Pool(lrng, nb)
    q = _normal_bits(vrng, (num_prompts * branches, num_q_heads, head_dim), src_dtype)
    pre_k = _normal_bits(vrng, (num_prompts, prefix_len, num_kv_heads, head_dim), src_dtype)
    pre_v = _normal_bits(vrng, (num_prompts, prefix_len, num_kv_heads, head_dim), src_dtype)
    rows, w1, w2, pairs, new = [], [], [], [], []
    tk, tv = [], []
    for p in range(num_prompts):
        shared_row = pool.take(pblk) if shared else None
        if shared:
            w1.append((pre_k[p], pre_v[p], slots_for(shared_row, np.arange(prefix_len), bs)))
        for b in range(branches):
            L = int(lens[p, b])
            if shared:
                row = shared_row.copy()
                if b > 0:                       # copy-on-write of the last prefix block
                    dst = pool.take(1)[0]
                    pairs.append((int(shared_row[-1]), int(dst)))
                    row[-1] = dst
            else:
                row = pool.take(pblk)
                w1.append((pre_k[p], pre_v[p], slots_for(row, np.arange(prefix_len), bs)))
            row = np.concatenate([row, pool.take(int(nblk[p, b]) - pblk)])
            rows.append(row)
            tail = L - prefix_len                  # tail tokens incl. the new one
            k_t = _normal_bits(vrng, (tail, num_kv_heads, head_dim), src_dtype)
            v_t = _normal_bits(vrng, (tail, num_kv_heads, head_dim), src_dtype)
            pos = np.arange(prefix_len, L)
            sl = slots_for(row, pos, bs)
            if tail > 1:
                w2.append((k_t[:-1], v_t[:-1], sl[:-1]))
            new.append((k_t[-1:], v_t[-1:], sl[-1:]))
    bt = _tables(rows, pool.pad)

    def cat(items):
        return WriteOp(np.concatenate([a for a, _, _ in items]), np.concatenate([b for _, b, _ in items]),
                       np.concatenate([c for _, _, c in items]))

    setup = [cat(w1)]
    if pairs:
        setup.append(CopyOp(np.asarray(pairs, dtype=np.int32)))
    if w2:
        setup.append(cat(w2))
    return PagedBatch(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      block_size=bs, src_dtype=src_dtype, kv_dtype=src_dtype, num_blocks=nb, pad_block=pool.pad,
                      block_tables=bt, seq_lens=lens.reshape(-1).astype(np.int32), q=q,
                      scale=float(np.float32(1.0) / np.sqrt(np.float32(head_dim))), setup=setup,
                      step_write=cat(new), blocks_unshared=unshared_need)


def mixed_prefill_batch(name: str = "chunked-prefill mixed batch, fp8 KV", chunk: int = 512, q_start: int = 4096,
                        num_decode: int = 128, dec_min: int = 256, dec_max: int = 8192, num_q_heads: int = 32,
                        num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16, src_dtype: str = "bf16",
                        kv_dtype: str = "fp8", seed: int = 4) -> PagedBatch:
    """One causal prefill chunk of ``chunk`` rows at positions q_start.. over
    its paged context, batched with ``num_decode`` decode sequences.  The
    chunk's own K/V and each decode sequence's new token are written inside
    the step; the older context is written in setup."""
    bs = block_size
    vrng = np.random.default_rng(seed)
    lrng = np.random.default_rng(seed + 1000)
    dlens = vrng.integers(dec_min, dec_max + 1, size=num_decode).astype(np.int64)
    plen = q_start + chunk
    need = int((-(-dlens // bs)).sum()) + -(-plen // bs)
    nb = _pool_size(need)
    pool = _Pool(lrng, nb)
    drows = [pool.take(int(-(-L // bs))) for L in dlens]
    prow = pool.take(-(-plen // bs))
    q_dec = _normal_bits(vrng, (num_decode, num_q_heads, head_dim), src_dtype)
    q_chk = _normal_bits(vrng, (chunk, num_q_heads, head_dim), src_dtype)
    dT = int(dlens.sum())
    dk = _normal_bits(vrng, (dT, num_kv_heads, head_dim), src_dtype)
    dv = _normal_bits(vrng, (dT, num_kv_heads, head_dim), src_dtype)
    pk = _normal_bits(vrng, (plen, num_kv_heads, head_dim), src_dtype)
    pv = _normal_bits(vrng, (plen, num_kv_heads, head_dim), src_dtype)
    dbt = _tables(drows, pool.pad)
    pbt = _tables([prow], pool.pad)
    dslots = np.concatenate([slots_for(dbt[i], np.arange(dlens[i]), bs) for i in range(num_decode)])
    pslots = slots_for(pbt[0], np.arange(plen), bs)
    starts = np.concatenate([[0], np.cumsum(dlens)[:-1]])
    is_new = np.zeros(dT, dtype=bool)
    is_new[starts + dlens - 1] = True
    setup = [WriteOp(np.concatenate([dk[~is_new], pk[:q_start]]), np.concatenate([dv[~is_new], pv[:q_start]]),
                     np.concatenate([dslots[~is_new], pslots[:q_start]]))]
    step = WriteOp(np.concatenate([pk[q_start:], dk[is_new]]), np.concatenate([pv[q_start:], dv[is_new]]),
                   np.concatenate([pslots[q_start:], dslots[is_new]]))
    if kv_dtype == "fp8":
        ks, vs = _fp8_scales([dk, pk], [dv, pv], src_dtype)
    else:
        ks, vs = 1.0, 1.0
    pre = PrefillPart(q=q_chk, cu_q_lens=np.array([0, chunk], dtype=np.int32),
                      q_start=np.array([q_start], dtype=np.int32), block_tables=pbt,
                      seq_lens=np.array([plen], dtype=np.int32))
    return PagedBatch(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      block_size=bs, src_dtype=src_dtype, kv_dtype=kv_dtype, num_blocks=nb, pad_block=pool.pad,
                      block_tables=dbt, seq_lens=dlens.astype(np.int32), q=q_dec,
                      scale=float(np.float32(1.0) / np.sqrt(np.float32(head_dim))), setup=setup, step_write=step,
                      prefill=pre, k_scale=ks, v_scale=vs, blocks_unshared=need)


def prefill_batch(name: str, chunks, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                  src_dtype: str = "bf16", kv_dtype: str | None = None, seed: int = 0,
                  fp8_scales: str = "tensor") -> PagedBatch:
    """Prefill-only batch: ``chunks`` is a list of (q_start, chunk_len).  The
    context 0..q_start-1 is written in setup, the chunk's own K/V in the step."""
    kv_dtype = kv_dtype or src_dtype
    bs = block_size
    vrng = np.random.default_rng(seed)
    lrng = np.random.default_rng(seed + 1000)
    lens = np.array([s + c for s, c in chunks], dtype=np.int64)
    need = int((-(-lens // bs)).sum())
    nb = _pool_size(need, round_to=64)
    pool = _Pool(lrng, nb)
    rows = [pool.take(int(-(-L // bs))) for L in lens]
    bt = _tables(rows, pool.pad)
    total = int(sum(c for _, c in chunks))
    q = _normal_bits(vrng, (total, num_q_heads, head_dim), src_dtype)
    ks, vs, kn, vn, sc, sn = [], [], [], [], [], []
    for i, (s, c) in enumerate(chunks):
        L = s + c
        k = _normal_bits(vrng, (L, num_kv_heads, head_dim), src_dtype)
        v = _normal_bits(vrng, (L, num_kv_heads, head_dim), src_dtype)
        sl = slots_for(bt[i], np.arange(L), bs)
        ks.append(k[:s]); vs.append(v[:s]); sc.append(sl[:s])
        kn.append(k[s:]); vn.append(v[s:]); sn.append(sl[s:])
    ctx = WriteOp(np.concatenate(ks), np.concatenate(vs), np.concatenate(sc))
    new = WriteOp(np.concatenate(kn), np.concatenate(vn), np.concatenate(sn))
    if kv_dtype == "fp8":
        k_scale, v_scale = _fp8_scales([ctx.k, new.k], [ctx.v, new.v], src_dtype, fp8_scales == "head")
    else:
        k_scale, v_scale = 1.0, 1.0
    cu = np.concatenate([[0], np.cumsum([c for _, c in chunks])]).astype(np.int32)
    pre = PrefillPart(q=q, cu_q_lens=cu, q_start=np.array([s for s, _ in chunks], dtype=np.int32),
                      block_tables=bt, seq_lens=lens.astype(np.int32))
    empty_bt = np.full((0, 1), pool.pad, dtype=np.int32)
    return PagedBatch(name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      block_size=bs, src_dtype=src_dtype, kv_dtype=kv_dtype, num_blocks=nb, pad_block=pool.pad,
                      block_tables=empty_bt, seq_lens=np.zeros(0, np.int32),
                      q=np.zeros((0, num_q_heads, head_dim), np.uint16),
                      scale=float(np.float32(1.0) / np.sqrt(np.float32(head_dim))), setup=[ctx], step_write=new,
                      prefill=pre, k_scale=k_scale, v_scale=v_scale, blocks_unshared=need)


# ------------------------------------------------------------- the five configs
def lognormal_lens(rng: np.random.Generator, n: int, median: float = 1000.0, sigma: float = 1.0,
                   cap: int = 8192) -> np.ndarray:
    """Context lengths log-normal with the given median; sigma is not given
    for this workload and is taken as 1.0; clipped to [1, cap]."""
    z = rng.standard_normal(n)
    return np.clip(np.rint(np.exp(np.log(median) + sigma * z)), 1, cap).astype(np.int64)


def cfg_tiny(seed: int = 0) -> PagedBatch:
    """1 layer, 4 sequences of 1/17/33/100 tokens, 4 q heads / 4 KV heads,
    head_dim 64, block 16, fp16, pool of 64 blocks."""
    return decode_batch("tiny paged decode", [1, 17, 33, 100], 4, 4, 64, 16, "f16", seed=seed,
                        num_blocks=64, scale=float(np.float32(0.125)))


def _fp8_name(kv_dtype: str, fp8_scales: str) -> str:
    if kv_dtype != "fp8":
        return ""
    return ", fp8 KV with per-head scales" if fp8_scales == "head" else ", fp8 KV"


def cfg_llama8b(seed: int = 1, batch: int = 64, kv_dtype: str = "bf16", fp8_scales: str = "tensor") -> PagedBatch:
    """Llama-3-8B-shaped decode layer: 32/8 heads, head_dim 128, block 16,
    bf16, lengths uniform 512..4096, 20k-block pool.  kv_dtype "fp8" stores
    the same values as e4m3 codes with per-tensor scales (fp8_scales "head":
    one scale per KV head)."""
    lens = np.random.default_rng(seed + 100).integers(512, 4097, size=batch)
    name = "Llama-3-8B-shaped decode layer" + _fp8_name(kv_dtype, fp8_scales)
    return decode_batch(name, lens, 32, 8, 128, 16, "bf16", kv_dtype=kv_dtype, seed=seed, num_blocks=20000,
                        fp8_scales=fp8_scales)


def cfg_llama70b(seed: int = 2, batch: int = 256, kv_dtype: str = "bf16", fp8_scales: str = "tensor") -> PagedBatch:
    """Llama-3-70B-shaped decode layer: 64/8 heads, head_dim 128, block 32,
    bf16, log-normal lengths (median 1000, cap 8192), split-KV 512.  kv_dtype
    "fp8" stores the same values as e4m3 codes with per-tensor scales
    (fp8_scales "head": one scale per KV head)."""
    lens = lognormal_lens(np.random.default_rng(seed + 100), batch)
    name = "Llama-3-70B-shaped decode layer" + _fp8_name(kv_dtype, fp8_scales)
    return decode_batch(name, lens, 64, 8, 128, 32, "bf16", kv_dtype=kv_dtype, seed=seed, partition_size=512,
                        fp8_scales=fp8_scales)


def cfg_d64(seed: int = 6, batch: int = 256, num_q_heads: int = 32, kv_dtype: str = "bf16") -> PagedBatch:
    """head_dim-64 decode layer: num_q_heads/8 heads (32/8: 4 query heads per KV
    head, 64/8: 8), block 16, bf16, lengths uniform 512..4096, split-KV 512,
    40k-block pool."""
    lens = np.random.default_rng(seed + 100).integers(512, 4097, size=batch)
    name = f"head_dim-64 decode layer, {num_q_heads}/8 heads" + _fp8_name(kv_dtype, "tensor")
    return decode_batch(name, lens, num_q_heads, 8, 64, 16, "bf16", kv_dtype=kv_dtype, seed=seed, num_blocks=40000,
                        partition_size=512)


def cfg_gqa(num_q_heads: int, seed: int = 7, batch: int = 128) -> PagedBatch:
    """Decode layer with num_q_heads/8 heads (groups such as 3 or 5 query heads
    per KV head), head_dim 128, block 16, bf16, lengths uniform 512..4096,
    split-KV 512, 40k-block pool."""
    lens = np.random.default_rng(seed + 100).integers(512, 4097, size=batch)
    return decode_batch(f"GQA decode layer, {num_q_heads}/8 heads", lens, num_q_heads, 8, 128, 16, "bf16", seed=seed,
                        num_blocks=40000, partition_size=512)


def cfg_shared_prefix(seed: int = 3, num_prompts: int = 32) -> PagedBatch:
    return shared_prefix_batch(num_prompts=num_prompts, seed=seed)


def cfg_mixed_fp8(seed: int = 4, num_decode: int = 128) -> PagedBatch:
    return mixed_prefill_batch(num_decode=num_decode, seed=seed)


# Prefill-only batches the benchmark times (and the tests compare in full):
# (description, builder).  Chunk sizes follow the pages' 512-token chunks and
# the 256 / 2048-token variants; one batch fills every SM with two-tile CTAs.
PREFILL_WORKLOADS = {
    "bf16_8x2048": ("8 chunks x 2048 tokens at position 2048, GQA 32/8, head_dim 128, block 16, bf16 KV",
                    lambda: prefill_batch("prefill 8x2048", [(2048, 2048)] * 8, 32, 8, 128, 16, "bf16", seed=3)),
    "bf16_chunk2048": ("one 2048-token chunk at position 4096, GQA 32/8, head_dim 128, block 16, bf16 KV",
                       lambda: prefill_batch("prefill chunk 2048", [(4096, 2048)], 32, 8, 128, 16, "bf16", seed=5)),
    "bf16_mha_4x1024": ("4 chunks x 1024 tokens at position 1024, MHA 32/32, head_dim 128, block 16, bf16 KV",
                        lambda: prefill_batch("prefill MHA 4x1024", [(1024, 1024)] * 4, 32, 32, 128, 16, "bf16",
                                              seed=6)),
    "bf16_16x256": ("16 chunks x 256 tokens at position 1024, GQA 32/8, head_dim 128, block 16, bf16 KV",
                    lambda: prefill_batch("prefill 16x256", [(1024, 256)] * 16, 32, 8, 128, 16, "bf16", seed=7)),
}


NAMED_WORKLOADS = {
    "tiny": cfg_tiny,
    "llama8b": cfg_llama8b,
    "llama70b": cfg_llama70b,
    "shared_prefix": cfg_shared_prefix,
    "mixed_fp8": cfg_mixed_fp8,
}


def empty_pools(b: PagedBatch):
    """Host K and V pools [NB, Hkv, bs, d] filled with the cache dtype's NaN bits."""
    shape = (b.num_blocks, b.num_kv_heads, b.block_size, b.head_dim)
    dt = np.uint8 if b.kv_dtype == "fp8" else np.uint16
    return np.full(shape, NAN_BITS[b.kv_dtype], dtype=dt), np.full(shape, NAN_BITS[b.kv_dtype], dtype=dt)
