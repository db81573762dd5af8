"""Pins of the oracle's paged attention (decode and chunked prefill).

The pages state that PagedAttention is exact: paging changes where K and V
live, not the result ("Inside vLLM Architecture", section "Semantic FAQ
Section").  So the oracle is pinned against (a) an independently written numpy
brute force over contiguous, unpaged K/V, (b) closed forms (one-token context,
constant V, zero query), and (c) invariances of the paged layout (block
permutation, block size, shared vs unshared prefix blocks, chunking).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from _brute import attention, causal_attention, decode_contiguous, to_f64


def _run_decode(b):
    kp, vp = W.empty_pools(b)
    oracle.populate(b, kp, vp)
    return oracle.decode_batch(b, kp, vp), kp, vp


@pytest.mark.parametrize("hq,hkv,d,bs,dt", [
    (4, 4, 64, 16, "f16"), (8, 2, 16, 16, "bf16"), (6, 3, 4, 32, "bf16"), (2, 1, 8, 16, "f16"),
])
def test_decode_vs_bruteforce(hq, hkv, d, bs, dt):
    lens = [1, 2, 15, 16, 17, 33, 40]
    b = W.decode_batch("t", lens, hq, hkv, d, bs, dt, seed=11)
    out, _, _ = _run_decode(b)
    for i, (K, V) in enumerate(decode_contiguous(b)):
        ref = attention(to_f64(b.q[i], dt), to_f64(K, dt), to_f64(V, dt), b.scale)
        np.testing.assert_allclose(out[i], ref, rtol=0, atol=1e-12)


def test_tiny_config_vs_bruteforce():
    b = W.cfg_tiny()
    out, _, _ = _run_decode(b)
    for i, (K, V) in enumerate(decode_contiguous(b)):
        ref = attention(to_f64(b.q[i], "f16"), to_f64(K, "f16"), to_f64(V, "f16"), b.scale)
        np.testing.assert_allclose(out[i], ref, rtol=0, atol=1e-12)


def test_single_token_context_returns_v():
    b = W.decode_batch("t", [1, 1, 1], 8, 2, 64, 16, "bf16", seed=3)
    out, _, _ = _run_decode(b)
    v = to_f64(b.step_write.v, "bf16")                       # [B, Hkv, d]
    assert np.array_equal(out, np.repeat(v, 4, axis=1))


def test_constant_v_returns_v():
    b = W.decode_batch("t", [5, 40, 77], 4, 2, 32, 16, "bf16", seed=4)
    c = W.round_to_bits(np.float32([0.71875]), "bf16")[0]
    for op in b.setup + [b.step_write]:
        op.v[...] = c
    out, _, _ = _run_decode(b)
    np.testing.assert_allclose(out, 0.71875, rtol=0, atol=1e-15)


def test_zero_query_gives_mean_of_v():
    b = W.decode_batch("t", [3, 31, 64], 4, 4, 16, 16, "f16", seed=5)
    b.q[...] = 0
    out, _, _ = _run_decode(b)
    for i, (K, V) in enumerate(decode_contiguous(b)):
        np.testing.assert_allclose(out[i], to_f64(V, "f16").mean(axis=0), rtol=0, atol=1e-12)


def test_gqa_head_mapping():
    """Query head h reads KV head h // (Hq/Hkv): zero all V heads but one and
    only that head's query group sees non-zero output."""
    b = W.decode_batch("t", [9, 20], 8, 4, 16, 16, "bf16", seed=6)
    for op in b.setup + [b.step_write]:
        op.v[:, [0, 1, 3], :] = 0
    out, _, _ = _run_decode(b)
    nz = np.abs(out).max(axis=(0, 2)) > 0
    assert nz.tolist() == [False, False, False, False, True, True, False, False]


def test_zero_length_sequence_gives_zero():
    b = W.decode_batch("t", [0, 5], 2, 2, 8, 16, "bf16", seed=7)
    out, _, _ = _run_decode(b)
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.isfinite(out[1]).all()


def test_block_permutation_and_block_size_invariance():
    lens = [1, 16, 17, 100, 257]
    ref, _, _ = _run_decode(W.decode_batch("t", lens, 8, 2, 32, 16, "bf16", seed=8))
    for layout_seed, bs in [(100, 16), (200, 16), (300, 32), (400, 32)]:
        got, _, _ = _run_decode(W.decode_batch("t", lens, 8, 2, 32, bs, "bf16", seed=8, layout_seed=layout_seed))
        assert np.array_equal(got, ref)


def test_shared_prefix_equals_unshared_copies():
    kw = dict(num_prompts=3, branches=4, prefix_len=64, tail_max=40, num_q_heads=4, num_kv_heads=2,
              head_dim=16, block_size=16, seed=9)
    sb = W.shared_prefix_batch(shared=True, **kw)
    ub = W.shared_prefix_batch(shared=False, **kw)
    assert sb.blocks_used() < ub.blocks_used()
    s, _, _ = _run_decode(sb)
    u, _, _ = _run_decode(ub)
    assert np.array_equal(s, u)
    assert np.isfinite(s).all()


def test_nan_pool_poisoning_is_never_read():
    """Every slot that no sequence owns holds NaN; a finite result shows the
    gather touched only owned slots."""
    b = W.decode_batch("t", [3, 19, 45], 4, 2, 16, 16, "bf16", seed=12)
    out, kp, _ = _run_decode(b)
    assert np.isfinite(out).all()
    assert (kp[b.pad_block] == W.NAN_BITS["bf16"]).all()


def _run_prefill(b):
    kp, vp = W.empty_pools(b)
    oracle.populate(b, kp, vp)
    return oracle.prefill_batch(b, kp, vp), kp, vp


def _prefill_contiguous(b, c):
    """Contiguous (K, V) bits of prefill chunk c of a ``prefill_batch``."""
    p = b.prefill
    ctx, new = b.setup[0], b.step_write
    starts = np.concatenate([[0], np.cumsum(p.q_start)])
    lens = np.diff(p.cu_q_lens)
    nstarts = np.concatenate([[0], np.cumsum(lens)])
    K = np.concatenate([ctx.k[starts[c]:starts[c + 1]], new.k[nstarts[c]:nstarts[c + 1]]])
    V = np.concatenate([ctx.v[starts[c]:starts[c + 1]], new.v[nstarts[c]:nstarts[c + 1]]])
    return K, V


@pytest.mark.parametrize("chunks", [[(0, 37)], [(50, 20), (0, 5), (17, 1)], [(16, 16), (33, 31)]])
def test_prefill_vs_bruteforce_causal(chunks):
    b = W.prefill_batch("p", chunks, 4, 2, 16, 16, "bf16", seed=13)
    out, _, _ = _run_prefill(b)
    p = b.prefill
    for c, (s, n) in enumerate(chunks):
        K, V = _prefill_contiguous(b, c)
        Q = to_f64(p.q[p.cu_q_lens[c]:p.cu_q_lens[c + 1]], "bf16")
        ref = causal_attention(Q, to_f64(K, "bf16"), to_f64(V, "bf16"), s, b.scale)
        np.testing.assert_allclose(out[p.cu_q_lens[c]:p.cu_q_lens[c + 1]], ref, rtol=0, atol=1e-12)


def test_prefill_last_row_equals_decode():
    b = W.prefill_batch("p", [(40, 9)], 8, 2, 32, 16, "f16", seed=14)
    out, kp, vp = _run_prefill(b)
    p = b.prefill
    dec = oracle.decode(p.q[-1:], oracle.F16, kp, vp, oracle.F16, p.block_tables, p.seq_lens, b.scale)
    assert np.array_equal(out[-1], dec[0])


def test_prefill_chunking_equals_one_shot():
    """A prompt processed as chunks [0,24) then [24,61) gives the same rows as
    one chunk [0,61): the rows see the same keys either way."""
    one = W.prefill_batch("p", [(0, 61)], 4, 4, 16, 16, "bf16", seed=15)
    out1, kp, vp = _run_prefill(one)
    p = one.prefill
    cu = np.array([0, 24, 61], np.int32)
    qs = np.array([0, 24], np.int32)
    bt = np.repeat(p.block_tables, 2, axis=0)
    out2 = oracle.prefill(p.q, oracle.BF16, cu, qs, kp, vp, oracle.BF16, bt, one.scale)
    assert np.array_equal(out1, out2)


def test_fp8_decode_uses_code_times_scale():
    """fp8 KV: each element is code * tensor scale; with one token the output
    is exactly the dequantised V row."""
    b = W.decode_batch("t", [1, 1], 4, 2, 16, 16, "bf16", kv_dtype="fp8", seed=16)
    out, kp, vp = _run_decode(b)
    blk = b.block_tables[:, 0]
    vrow = oracle.e4m3_to_f64(vp[blk, :, 0, :]) * np.float64(np.float32(b.v_scale))
    assert np.array_equal(out, np.repeat(vrow, 2, axis=1))


def test_fp8_decode_close_to_bf16_decode():
    """The fp8 cache is a quantisation of the bf16 values: the two oracle
    results differ by about the e4m3 step (2^-4 relative), far below 1."""
    lens = [30, 64, 129]
    a, _, _ = _run_decode(W.decode_batch("t", lens, 8, 2, 64, 16, "bf16", seed=17))
    f, _, _ = _run_decode(W.decode_batch("t", lens, 8, 2, 64, 16, "bf16", kv_dtype="fp8", seed=17))
    err = np.abs(a - f).max()
    assert 1e-4 < err < 0.1
