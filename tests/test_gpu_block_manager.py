"""The host block manager feeding the kernels, end to end on the GPU.

A batch of prompts is laid out by pa_bm_* (seeded shuffled pool), forked
into branches that append different numbers of tokens (copy-on-write of a
shared partial last block, "High-Throughput LLM Serving with vLLM &
PagedAttention", section "2. Virtual Memory Paging Applied to GPUs"), and
a second copy of one prompt is matched against the prefix cache (its full
blocks get slot -1 and are not written again).  The GPU runs write ->
copy_blocks -> write -> decode through the C ABI; the oracle runs its own
write, copy and decode on host pools from the same slots, pairs and block
tables.  Pools must agree bit for bit, outputs within the decode
tolerance."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_writes_gb300 as pa
import workloads as W
from paged_kv_cache_writes_gb300.staging import to_bits, to_device
from _gpu import TOL, max_err

pytestmark = pytest.mark.gpu


def _pools(nb, hkv, bs, d, kv):
    shape = (nb, hkv, bs, d)
    dt = np.uint8 if kv == "fp8" else np.uint16
    k = np.full(shape, W.NAN_BITS[kv], dtype=dt)
    return k, k.copy()


@pytest.mark.parametrize("kv,src", [("bf16", "bf16"), ("f16", "f16"), ("fp8", "bf16")])
@pytest.mark.parametrize("bs", [16, 32])
def test_forked_batch_through_the_block_manager(kv, src, bs):
    hq, hkv, d, nb = 32, 8, 128, 512
    k_scale, v_scale = (0.5, 0.75) if kv == "fp8" else (1.0, 1.0)
    rng = np.random.default_rng(1000 + bs)
    bm = pa.BlockManager(nb, bs, shuffle_seed=17)

    # phase 1: prompts (ragged, mostly not block-aligned), one of them with token ids
    prompt_lens = [3 * bs + 5, 1, 2 * bs, 5 * bs + bs - 1, 7]
    ids0 = rng.integers(0, 32000, size=prompt_lens[0]).astype(np.int32)
    parents, slots1 = [], []
    for i, L in enumerate(prompt_lens):
        s = bm.new_sequence()
        slots, cow = bm.append(s, L, ids0 if i == 0 else None)
        assert len(cow) == 0
        parents.append(s)
        slots1.append(slots)
    # a second copy of prompt 0: its full blocks come from the prefix cache
    twin = bm.new_sequence()
    twin_slots, _ = bm.append(twin, len(ids0), ids0)
    nfull = len(ids0) // bs
    assert (twin_slots[:nfull * bs] == -1).all() and (twin_slots[nfull * bs:] >= 0).all()
    k1 = W._normal_bits(rng, (sum(prompt_lens), hkv, d), src)
    v1 = W._normal_bits(rng, (sum(prompt_lens), hkv, d), src)
    # the twin's tokens carry the same K/V as prompt 0's (same ids, same prefix)
    k1 = np.concatenate([k1, k1[:len(ids0)]])
    v1 = np.concatenate([v1, v1[:len(ids0)]])
    slot1 = np.concatenate(slots1 + [twin_slots])

    # phase 2: three forks per prompt; every sequence (parents too) appends a ragged number of tokens
    seqs, slots2, pairs = list(parents) + [twin], [], []
    for p in parents:
        seqs += [bm.fork(p) for _ in range(3)]
    for s in seqs:
        slots, cow = bm.append(s, int(rng.integers(1, 2 * bs + 3)))
        slots2.append(slots)
        pairs += cow.tolist()
    assert len(pairs) >= 4                                   # copy-on-write happened
    slot2 = np.concatenate(slots2)
    k2 = W._normal_bits(rng, (len(slot2), hkv, d), src)
    v2 = W._normal_bits(rng, (len(slot2), hkv, d), src)
    pairs = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)

    tables = [bm.block_table(s) for s in seqs]
    max_blocks = max(len(t) for t, _ in tables)
    block_tables = np.full((len(seqs), max_blocks), -1, dtype=np.int32)
    for i, (t, _) in enumerate(tables):
        block_tables[i, :len(t)] = t
    seq_lens = np.asarray([L for _, L in tables], dtype=np.int32)
    q = W._normal_bits(rng, (len(seqs), hq, d), src)
    scale = d ** -0.5

    # oracle: its own write, copy, write, decode on host pools
    kvc, sc = oracle.DTYPE_CODES[kv], oracle.DTYPE_CODES[src]
    kp, vp = _pools(nb, hkv, bs, d, kv)
    oracle.reshape_and_cache(k1, v1, sc, slot1, kp, vp, kvc, k_scale, v_scale)
    oracle.copy_blocks(kp, vp, pairs)
    oracle.reshape_and_cache(k2, v2, sc, slot2, kp, vp, kvc, k_scale, v_scale)
    ref = oracle.decode(q, sc, kp, vp, kvc, block_tables, seq_lens, scale, k_scale, v_scale)

    # GPU: the same calls through the C ABI
    dev = torch.device("cuda")
    kc0, vc0 = _pools(nb, hkv, bs, d, kv)
    kc, vc = to_device(kc0, kv, dev), to_device(vc0, kv, dev)
    desc = pa.kv_cache_desc(kc, k_scale, v_scale)
    i64 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(dev)
    pa.pa_reshape_and_cache(to_device(k1, src, dev), to_device(v1, src, dev), i64(slot1), kc, vc, desc)
    pa.pa_copy_blocks(kc, vc, desc, torch.from_numpy(pairs).to(dev))
    pa.pa_reshape_and_cache(to_device(k2, src, dev), to_device(v2, src, dev), i64(slot2), kc, vc, desc)
    qd = to_device(q, src, dev)
    out = torch.empty(qd.shape, dtype=torch.float32, device=dev)
    ws_bytes = pa.pa_decode_workspace_bytes(len(seqs), hq, hkv, d, int(seq_lens.max()), 256)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    pa.pa_decode(qd, kc, vc, desc, torch.from_numpy(block_tables).to(dev), torch.from_numpy(seq_lens).to(dev),
                 int(seq_lens.max()), scale, out, ws, 256)
    torch.cuda.synchronize()

    assert np.array_equal(to_bits(kc), kp) and np.array_equal(to_bits(vc), vp)
    err = max_err(out, ref)
    assert err <= TOL[kv], err
    # the twin attends to exactly what prompt 0's sequence held before its append
    assert seq_lens[len(parents)] > len(ids0)
    np.testing.assert_array_equal(block_tables[len(parents), :nfull], block_tables[0, :nfull])
