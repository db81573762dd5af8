"""fp8 caches with one scale per KV head, in the oracle.

A head's scale is read here as the per-tensor rule applied to that head's
values alone (amax over the head's K, resp. V, / 448).  Pins: head h of a
per-head write holds exactly the codes a per-tensor write with scale s_h
stores; a one-token context returns V's code times v_scale[h] exactly; and
decode / prefill with per-head scales equal, head group by head group, the
per-tensor runs with that head's scale."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")


def test_per_head_scales_follow_the_per_tensor_rule_head_by_head():
    b = W.decode_batch("hs", [40, 70, 129], 8, 4, 64, 16, "bf16", kv_dtype="fp8", seed=3, fp8_scales="head")
    k_all = np.concatenate([op.k for op in b.setup] + [b.step_write.k])
    for h in range(4):
        amax = W._amax(k_all[:, h, :], "bf16")
        assert b.k_scale[h] == np.float32(amax) / np.float32(448.0)
    assert len(set(b.k_scale.tolist())) > 1          # heads differ


def test_per_head_write_equals_per_tensor_writes_of_each_head():
    b = W.decode_batch("hs", [40, 70, 129], 8, 4, 64, 16, "bf16", kv_dtype="fp8", seed=4, fp8_scales="head")
    kp, vp = W.empty_pools(b)
    oracle.populate(b, kp, vp)
    for h in range(4):
        kh, vh = W.empty_pools(b)
        for op in list(b.setup) + [b.step_write]:
            oracle.reshape_and_cache(op.k, op.v, oracle.DTYPE_CODES["bf16"], op.slots, kh, vh,
                                     oracle.DTYPE_CODES["fp8"], float(b.k_scale[h]), float(b.v_scale[h]))
        assert np.array_equal(kp[:, h], kh[:, h]) and np.array_equal(vp[:, h], vh[:, h])


def test_one_token_context_returns_v_code_times_its_head_scale():
    b = W.decode_batch("hs1", [1, 1, 1], 8, 4, 64, 16, "bf16", kv_dtype="fp8", seed=5, fp8_scales="head")
    kp, vp = W.empty_pools(b)
    oracle.populate(b, kp, vp)
    out = oracle.decode_batch(b, kp, vp)
    for i in range(3):
        blk = b.block_tables[i][0]
        for hq in range(8):
            g = hq // 2
            codes = torch.from_numpy(np.ascontiguousarray(vp[blk, g, 0]))
            values = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()   # an independent e4m3 decoder
            want = values * np.float64(np.float32(b.v_scale[g]))
            np.testing.assert_array_equal(out[i, hq], want)


def test_per_head_decode_and_prefill_equal_per_tensor_runs_by_group():
    b = W.decode_batch("hsd", [33, 300, 1000], 8, 4, 64, 16, "bf16", kv_dtype="fp8", seed=6, fp8_scales="head")
    kp, vp = W.empty_pools(b)
    oracle.populate(b, kp, vp)
    out = oracle.decode_batch(b, kp, vp)
    for g in range(4):
        ref = oracle.decode(b.q, oracle.DTYPE_CODES["bf16"], kp, vp, oracle.DTYPE_CODES["fp8"], b.block_tables,
                            b.seq_lens, b.scale, float(b.k_scale[g]), float(b.v_scale[g]))
        np.testing.assert_array_equal(out[:, 2 * g:2 * g + 2], ref[:, 2 * g:2 * g + 2])
    p = W.prefill_batch("hsp", [(100, 37), (0, 64)], 8, 4, 64, 16, "bf16", kv_dtype="fp8", seed=7, fp8_scales="head")
    kp, vp = W.empty_pools(p)
    oracle.populate(p, kp, vp)
    out = oracle.prefill_batch(p, kp, vp)
    for g in range(4):
        pp = p.prefill
        ref = oracle.prefill(pp.q, oracle.DTYPE_CODES["bf16"], pp.cu_q_lens, pp.q_start, kp, vp,
                             oracle.DTYPE_CODES["fp8"], pp.block_tables, p.scale, float(p.k_scale[g]),
                             float(p.v_scale[g]))
        np.testing.assert_array_equal(out[:, 2 * g:2 * g + 2], ref[:, 2 * g:2 * g + 2])
