"""Host block manager (pa_bm_*): block tables, slots, fork / copy-on-write and
prefix reuse, checked against the pages' addressing and block arithmetic.

Slot of position p = table[p // bs] * bs + p % bs ("Inside vLLM Architecture",
"The Block Table Mapping Subsystem"); blocks are taken on demand, so a
sequence wastes fewer than bs slots ("Inside vLLM v0.7", "Architectural
Blueprint 2"; "High-Throughput LLM Serving", "2. Virtual Memory Paging Applied
to GPUs": under 4% waste, copy-on-write of shared blocks)."""
import numpy as np
import pytest

import paged_kv_cache_writes_gb300 as pa


def _slots_from_table(table, positions, bs):
    positions = np.asarray(positions, dtype=np.int64)
    return table[positions // bs].astype(np.int64) * bs + positions % bs


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("seed", [0, 7])
def test_slots_follow_the_block_table(bs, seed):
    bm = pa.BlockManager(512, bs, shuffle_seed=seed)
    rng = np.random.default_rng(3)
    seqs = {bm.new_sequence(): 0 for _ in range(5)}
    history = {s: [] for s in seqs}
    for _ in range(40):                      # interleaved appends of ragged sizes
        s = int(rng.choice(list(seqs)))
        n = int(rng.integers(0, 3 * bs))
        slots, cow = bm.append(s, n)
        assert len(cow) == 0
        history[s].extend(slots.tolist())
        seqs[s] += n
    used = set()
    for s, L in seqs.items():
        table, length = bm.block_table(s)
        assert length == L
        assert len(table) == -(-L // bs)                        # blocks on demand
        assert np.array_equal(np.asarray(history[s]), _slots_from_table(table, np.arange(L), bs))
        assert not used & set(table.tolist())                   # no block belongs to two sequences
        used |= set(table.tolist())
    st = bm.stats()
    assert st.used_blocks == len(used) and st.free_blocks == 512 - len(used)
    assert st.logical_tokens == sum(seqs.values())


def test_shuffled_pool_is_a_seeded_permutation():
    a, b, c = (pa.BlockManager(256, 16, shuffle_seed=s) for s in (5, 5, 6))
    ta, tb, tc = (m.append(m.new_sequence(), 256 * 16)[0] // 16 for m in (a, b, c))
    blocks_a = ta[::16]
    assert sorted(blocks_a.tolist()) == list(range(256))
    assert np.array_equal(ta, tb) and not np.array_equal(ta, tc)
    plain = pa.BlockManager(8, 16)
    assert (plain.append(plain.new_sequence(), 128)[0][::16] // 16).tolist() == list(range(8))


def test_waste_under_four_percent_on_decode_lengths():
    # Llama-3-8B-shaped decode lengths: uniform 512..4096 tokens, blocks of 16
    lens = np.random.default_rng(101).integers(512, 4097, size=64)
    bm = pa.BlockManager(20000, 16)
    for L in lens:
        bm.append(bm.new_sequence(), int(L))
    st = bm.stats()
    slots = st.used_blocks * 16
    assert st.logical_tokens == lens.sum()
    assert slots - st.logical_tokens < 16 * len(lens)          # < one block per sequence
    assert (slots - st.logical_tokens) / slots < 0.04


@pytest.mark.parametrize("prefix", [40, 48])
def test_fork_shares_blocks_and_copies_a_shared_partial_block_once(prefix):
    bs = 16
    bm = pa.BlockManager(64, bs)
    parent = bm.new_sequence()
    bm.append(parent, prefix)
    ptable, _ = bm.block_table(parent)
    kids = [bm.fork(parent) for _ in range(3)]
    st = bm.stats()
    assert st.used_blocks == len(ptable) and st.shared_blocks == len(ptable)
    for i, k in enumerate(kids):
        slots, cow = bm.append(k, 5 + i)
        table, L = bm.block_table(k)
        assert L == prefix + 5 + i
        if prefix % bs:                                          # shared partial last block: one copy
            assert cow.tolist() == [[ptable[-1], table[len(ptable) - 1]]]
            assert table[len(ptable) - 1] != ptable[-1]
            assert np.array_equal(table[:len(ptable) - 1], ptable[:-1])
        else:                                                    # block-aligned: nothing to copy
            assert len(cow) == 0
            assert np.array_equal(table[:len(ptable)], ptable)
        assert np.array_equal(slots, _slots_from_table(table, np.arange(prefix, L), bs))
        slots2, cow2 = bm.append(k, 3)                           # the copy is private now
        assert len(cow2) == 0
    # the parent still owns its original last block
    assert np.array_equal(bm.block_table(parent)[0], ptable)
    for s in kids + [parent]:
        bm.free(s)
    st = bm.stats()
    assert st.free_blocks == 64 and st.used_blocks == 0 and st.shared_blocks == 0


def test_shared_prefix_saving_matches_block_arithmetic():
    # 32 prompts x 4 branches, 2048-token shared prefix (128 blocks of 16), tails uniform 0..256
    rng = np.random.default_rng(11)
    bs, prefix = 16, 2048
    tails = rng.integers(0, 257, size=(32, 4))
    bm = pa.BlockManager(8192, bs, shuffle_seed=1)
    for p in range(32):
        root = bm.new_sequence()
        bm.append(root, prefix)
        branches = [root] + [bm.fork(root) for _ in range(3)]
        for b, s in enumerate(branches):
            bm.append(s, int(tails[p, b]))
    st = bm.stats()
    unshared = int(sum(-(-(prefix + t) // bs) for t in tails.ravel()))
    shared = 32 * (prefix // bs) + int(sum(-(-t // bs) for t in tails.ravel()))
    assert st.logical_blocks == unshared
    assert st.used_blocks == shared
    assert st.shared_blocks == 32 * (prefix // bs)
    saving = 1 - shared / unshared
    assert 0.65 < saving < 0.75


def test_out_of_blocks_leaves_state_unchanged():
    bm = pa.BlockManager(4, 16)
    s = bm.new_sequence()
    bm.append(s, 50)                                             # 4 blocks
    before = bm.block_table(s)
    with pytest.raises(pa.PaError) as e:
        bm.append(s, 20)
    assert e.value.status == 6                                   # PA_ERR_NO_BLOCKS
    after = bm.block_table(s)
    assert np.array_equal(before[0], after[0]) and before[1] == after[1]
    bm.append(s, 14)                                             # fills the last block: no new block
    assert bm.block_table(s)[1] == 64


def test_prefix_reuse_shares_only_identical_prefixes():
    bs = 16
    bm = pa.BlockManager(128, bs)
    rng = np.random.default_rng(5)
    ids = rng.integers(0, 32000, size=5 * bs + 7).astype(np.int32)
    a = bm.new_sequence()
    sa, _ = bm.append(a, len(ids), ids)
    assert (sa >= 0).all()
    assert bm.stats().cached_blocks == 5                          # full blocks only
    ta, _ = bm.block_table(a)
    # same ids: the 5 full blocks are shared (slots -1: already cached), the tail is new
    b = bm.new_sequence()
    sb, _ = bm.append(b, len(ids), ids)
    tb, _ = bm.block_table(b)
    assert (sb[:5 * bs] == -1).all() and (sb[5 * bs:] >= 0).all()
    assert np.array_equal(tb[:5], ta[:5]) and tb[5] != ta[5]
    # same ids after a different first block: nothing after the difference is shared
    ids2 = ids.copy()
    ids2[3] += 1
    c = bm.new_sequence()
    sc, _ = bm.append(c, len(ids2), ids2)
    assert (sc >= 0).all()
    assert not set(bm.block_table(c)[0].tolist()) & set(ta.tolist())
    # the second block's ids at position 0: different prefix, not shared
    d = bm.new_sequence()
    sd, _ = bm.append(d, bs, ids[bs:2 * bs])
    assert (sd >= 0).all() and bm.block_table(d)[0][0] not in ta.tolist()
    # appends without ids are never matched and never cached
    e = bm.new_sequence()
    se, _ = bm.append(e, 2 * bs)
    assert (se >= 0).all()
    # a shared cached block outlives its first owner; it leaves the cache with its last reference
    bm.free(a)
    assert set(ta[:5].tolist()) <= set(bm.block_table(b)[0].tolist())
    bm.free(b)
    st = bm.stats()
    assert all(blk not in bm.block_table(c)[0].tolist() for blk in ta[:5])
    # left in the cache: c's 5 full blocks and d's one (a's and b's shared blocks went with their last owner)
    assert st.cached_blocks == 5 + 1


def test_invalid_arguments():
    with pytest.raises(pa.PaError):
        pa.BlockManager(0, 16)
    bm = pa.BlockManager(8, 16)
    with pytest.raises(pa.PaError):
        bm.append(3, 1)                                          # unknown sequence
    s = bm.new_sequence()
    bm.free(s)
    with pytest.raises(pa.PaError):
        bm.append(s, 1)                                          # freed sequence
    with pytest.raises(pa.PaError):
        bm.fork(s)
