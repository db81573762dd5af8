"""Host side of the fused and mixed steps (no GPU): the staging layer splits a
step's new tokens into each decode row's token at the slot of its last
position (stored by pa_decode_write / pa_mixed_step) and the rest (the
prefill chunk's own tokens, written first), and the two parts together are
exactly the step's writes."""
import numpy as np

import workloads as W
from paged_kv_cache_writes_gb300.staging import DeviceBatch, to_bits


def test_mixed_step_tokens_split_into_decode_rows_and_the_chunk():
    b = W.mixed_prefill_batch("split", chunk=50, q_start=60, num_decode=7, dec_min=1, dec_max=300, seed=3)
    dev = DeviceBatch(b, "cpu")
    k, v, slots = dev.fused_step_tensors(allow_others=True)
    ok, ov, oslots = dev._others
    sw = b.step_write
    slots, oslots = slots.numpy(), oslots.numpy()
    # each decode row's token sits at the slot of its last position
    for i, L in enumerate(b.seq_lens):
        last = int(b.block_tables[i][(L - 1) // b.block_size]) * b.block_size + (L - 1) % b.block_size
        assert slots[i] == last
    # the two parts are the step's writes, each once, with their K/V
    got = np.concatenate([slots, oslots])
    assert sorted(got.tolist()) == sorted(sw.slots.tolist())
    by_slot = {int(s): t for t, s in enumerate(sw.slots)}
    k_all = np.concatenate([to_bits(k), to_bits(ok)])
    v_all = np.concatenate([to_bits(v), to_bits(ov)])
    for j, s in enumerate(got):
        assert np.array_equal(k_all[j], sw.k[by_slot[int(s)]]) and np.array_equal(v_all[j], sw.v[by_slot[int(s)]])
    # the chunk's own tokens are the rest: positions q_start .. q_start + chunk - 1 of the prefill sequence
    assert len(oslots) == 50


def test_decode_only_step_has_no_other_tokens():
    b = W.decode_batch("fused", [1, 17, 300], 8, 2, 64, 16, "f16", seed=4)
    dev = DeviceBatch(b, "cpu")
    dev.fused_step_tensors()
    assert dev._others is None
