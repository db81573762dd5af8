"""Pins of the oracle's cache write and block copy, and of the block manager's
slot arithmetic that feeds them.

Cache layout: pools [num_blocks][num_kv_heads][block_size][head_dim]; token t
with slot s goes to block s // block_size, offset s % block_size ("Inside vLLM
Architecture", section "The Block Table Mapping Subsystem", allocate_slot).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_golden_block_table_slots():
    for name, frames, pos, slot in _rows("block_table_examples.txt"):
        row = np.array([int(x) for x in frames.split(",")], dtype=np.int32)
        assert W.slots_for(row, [int(pos)], 16)[0] == int(slot), name


class _PageManager:
    """Restatement of the page's PagedKVCacheManager semantics (section "The
    Block Table Mapping Subsystem"): a new physical block is popped from the
    front of the free list whenever a token lands at offset 0."""

    def __init__(self, block_size, free):
        self.bs, self.free, self.tables = block_size, list(free), {}

    def allocate_slot(self, rid, seq_len):
        logical, offset = seq_len // self.bs, seq_len % self.bs
        self.tables.setdefault(rid, [])
        if offset == 0:
            self.tables[rid].append(self.free.pop(0))
        return self.tables[rid][logical]


def test_slots_follow_allocate_slot():
    b = W.decode_batch("t", [1, 16, 17, 40], 2, 2, 8, 16, "bf16", seed=1, num_blocks=64)
    bs = b.block_size
    # the free list the workload drew its blocks from, in hand-out order
    order = [int(x) for r, L in zip(b.block_tables, b.seq_lens) for x in r[:-(-L // bs)]]
    mgr = _PageManager(bs, order)
    slots = np.concatenate([b.setup[0].slots, b.step_write.slots])
    want = []
    for i, L in enumerate(b.seq_lens.tolist()):
        for p in range(L):
            want.append((mgr.allocate_slot(i, p), p % bs))
    ctx_slots = list(b.setup[0].slots)
    new_slots = list(b.step_write.slots)
    got, c = [], 0
    for i, L in enumerate(b.seq_lens.tolist()):
        got += ctx_slots[c:c + L - 1] + [new_slots[i]]
        c += L - 1
    assert len(got) == len(slots)
    assert [(s // bs, s % bs) for s in got] == want


def test_cache_write_layout_explicit():
    """Every written element lands at [slot//bs][h][slot%bs][e]; everything
    else keeps its previous bits; negative slots are skipped."""
    rng = np.random.default_rng(2)
    nb, hkv, bs, d, T = 7, 3, 16, 8, 12
    k = rng.integers(0, 1 << 16, size=(T, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(T, hkv, d), dtype=np.uint16)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[3] = -1
    kc = np.full((nb, hkv, bs, d), 0xABCD, np.uint16)
    vc = np.full((nb, hkv, bs, d), 0x1234, np.uint16)
    oracle.reshape_and_cache(k, v, oracle.BF16, slots, kc, vc, oracle.BF16)
    kw = np.full_like(kc, 0xABCD)
    vw = np.full_like(vc, 0x1234)
    for t in range(T):
        if slots[t] < 0:
            continue
        for h in range(hkv):
            for e in range(d):
                kw[slots[t] // bs, h, slots[t] % bs, e] = k[t, h, e]
                vw[slots[t] // bs, h, slots[t] % bs, e] = v[t, h, e]
    assert np.array_equal(kc, kw) and np.array_equal(vc, vw)


def test_cache_write_fp8_vs_torch_cast():
    """fp8 cache write = e4m3_rne_satfinite(fp32(x) / scale): checked against
    numpy's IEEE fp32 division followed by PyTorch's e4m3fn cast (in range)."""
    rng = np.random.default_rng(3)
    nb, hkv, bs, d, T = 5, 2, 16, 16, 30
    x = rng.standard_normal((T, hkv, d)).astype(np.float32) * 3
    kb = W.round_to_bits(x, "bf16")
    vb = W.round_to_bits(-x * 0.5, "bf16")
    ks = np.float32(np.abs(W.bits_to_f32(kb, "bf16")).max()) / np.float32(448)
    vs = np.float32(np.abs(W.bits_to_f32(vb, "bf16")).max()) / np.float32(448)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    kc = np.zeros((nb, hkv, bs, d), np.uint8)
    vc = np.zeros((nb, hkv, bs, d), np.uint8)
    oracle.reshape_and_cache(kb, vb, oracle.BF16, slots, kc, vc, oracle.FP8_E4M3, float(ks), float(vs))
    for src, sc, cache in ((kb, ks, kc), (vb, vs, vc)):
        q = W.bits_to_f32(src, "bf16") / np.float32(sc)
        assert q.dtype == np.float32 and np.abs(q).max() <= 448
        ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = cache[slots // bs, :, slots % bs, :]
        assert np.array_equal(got, ref)
    # the amax element maps to exactly +-448
    assert 0x7E in (kc & 0x7F)


def test_cache_write_f16_bits_unchanged():
    rng = np.random.default_rng(4)
    k = rng.integers(0, 1 << 16, size=(4, 1, 4), dtype=np.uint16)
    kc = np.zeros((2, 1, 16, 4), np.uint16)
    vc = np.zeros_like(kc)
    oracle.reshape_and_cache(k, k, oracle.F16, np.array([0, 5, 16, 31]), kc, vc, oracle.F16)
    assert np.array_equal(kc[0, 0, 0], k[0, 0]) and np.array_equal(kc[1, 0, 15], k[3, 0])


def test_cache_write_rejects_out_of_range_slot():
    kc = np.zeros((2, 1, 16, 4), np.uint16)
    k = np.zeros((1, 1, 4), np.uint16)
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(k, k, oracle.BF16, np.array([32]), kc, kc.copy(), oracle.BF16)


def test_copy_blocks_bitwise():
    rng = np.random.default_rng(5)
    kc = rng.integers(0, 1 << 16, size=(8, 2, 16, 4), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(8, 2, 16, 4), dtype=np.uint16)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[1, 6], [3, 0], [1, 7]], np.int32)
    oracle.copy_blocks(kc, vc, pairs)
    for s, d in pairs:
        assert np.array_equal(kc[d], k0[s]) and np.array_equal(vc[d], v0[s])
    for blk in (1, 2, 3, 4, 5):
        assert np.array_equal(kc[blk], k0[blk]) and np.array_equal(vc[blk], v0[blk])


def test_golden_kv_bytes_per_token():
    for name, hkv, d, eb, want in _rows("kv_bytes_per_token.txt"):
        b = W.decode_batch("t", [1], int(hkv), int(hkv), int(d), 16, "bf16", seed=0)
        assert b.decode_kv_bytes() == int(want), name
    # the 70B figure over 80 layers, against the page's doubled 655,360
    assert 4096 * 80 == 655360 // 2


def test_config_shapes():
    t = W.cfg_tiny()
    assert t.seq_lens.tolist() == [1, 17, 33, 100] and t.num_blocks == 64
    assert (t.num_q_heads, t.num_kv_heads, t.head_dim, t.block_size, t.kv_dtype) == (4, 4, 64, 16, "f16")
    assert t.blocks_used() == 1 + 2 + 3 + 7
