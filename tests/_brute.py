"""Independent numpy fp64 brute force for pinning the oracle.

Unpaged, vectorised attention over contiguous K/V, written without the
oracle's gather or loops: the GQA mapping is an explicit ``np.repeat`` of the
KV heads, softmax is evaluated with a max shift, and the causal case uses a
mask matrix.  Nothing here is imported by the oracle or by the product.
"""
import numpy as np

from workloads import bits_to_f32


def to_f64(bits, dtype):
    return bits_to_f32(np.ascontiguousarray(bits), dtype).astype(np.float64)


def attention(q, K, V, scale):
    """q [Hq, d]; K, V [L, Hkv, d] (fp64). Returns [Hq, d]."""
    hq, hkv = q.shape[0], K.shape[1]
    if K.shape[0] == 0:
        return np.zeros_like(q)
    Kr = np.repeat(K, hq // hkv, axis=1)
    Vr = np.repeat(V, hq // hkv, axis=1)
    s = np.einsum("hd,lhd->hl", q, Kr) * scale
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=1, keepdims=True)
    return np.einsum("hl,lhd->hd", w, Vr)


def causal_attention(Q, K, V, q_start, scale):
    """Q [n, Hq, d] at positions q_start..q_start+n-1; K, V [q_start+n, Hkv, d]."""
    n, hq, _ = Q.shape
    L, hkv, _ = K.shape
    Kr = np.repeat(K, hq // hkv, axis=1)
    Vr = np.repeat(V, hq // hkv, axis=1)
    s = np.einsum("nhd,lhd->nhl", Q, Kr) * scale
    pos = q_start + np.arange(n)[:, None]
    mask = np.arange(L)[None, :] <= pos
    s = np.where(mask[:, None, :], s, -np.inf)
    s = s - s.max(axis=2, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=2, keepdims=True)
    return np.einsum("nhl,lhd->nhd", w, Vr)


def decode_contiguous(batch):
    """Per-sequence contiguous (K, V) bits of a ``workloads.decode_batch``:
    the context rows come in sequence order, then each sequence's new row."""
    ctx = batch.setup[0]
    out, c, j = [], 0, 0
    for L in batch.seq_lens.tolist():
        if L == 0:
            out.append((ctx.k[:0], ctx.v[:0]))
            continue
        n = L - 1
        K = np.concatenate([ctx.k[c:c + n], batch.step_write.k[j:j + 1]])
        V = np.concatenate([ctx.v[c:c + n], batch.step_write.v[j:j + 1]])
        out.append((K, V))
        c += n
        j += 1
    return out
