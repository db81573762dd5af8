"""The operand split of the tensor-core decode on fp8 caches, checked
exhaustively on the CPU.

Its MMAs multiply the cache's e4m3 codes as stored, so the queries (scaled by
a power of two so that a unit's largest |q| lies in [128, 256)) enter as a sum
of e4m3 terms, each the nearest-even rounding of what the previous ones
leave: x = hi + lo/16 for bf16 queries, x = hi + mid/16 + lo/256 for f16
ones.  Restated here with PyTorch's e4m3 cast over every finite bf16 and f16
value with |x| <= 256:
  * two terms hold every bf16 value with |x| >= 2^-6 exactly, and any bf16
    value to 2^-14;
  * two terms do not hold f16 values (up to 2^-8 relative is lost), which is
    why f16 queries take three;
  * three terms hold every f16 value with |x| >= 2^-7 exactly, and any f16
    value to 2^-18.
The scale puts a unit's largest element in [128, 256), so the exact ranges
cover every element within 2^-13 (bf16) or 2^-14 (f16) of that largest one."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _e4m3(x):
    t = torch.from_numpy(np.clip(np.asarray(x, dtype=np.float32), -448, 448))
    return t.to(torch.float8_e4m3fn).to(torch.float32).numpy()


def _split(x, terms):
    x = np.asarray(x, dtype=np.float32)
    total = np.zeros(x.shape, np.float64)
    r, w = x, 1.0
    for _ in range(terms):
        c = _e4m3(r)
        total += c.astype(np.float64) * w
        r = ((r - c) * 16).astype(np.float32)   # exact: r - c has at most 8 significant bits here
        w /= 16
    return total


def _all(kind):
    if kind == "bf16":
        x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    else:
        x = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    return x[np.isfinite(x) & (np.abs(x) <= 256)]


def test_two_terms_hold_every_bf16_value():
    x = _all("bf16")
    err = np.abs(_split(x, 2) - x)
    assert err[np.abs(x) >= 2.0 ** -6].max() == 0
    assert err.max() <= 2.0 ** -14


def test_two_terms_lose_f16_bits():
    x = _all("f16")
    err = np.abs(_split(x, 2) - x)
    big = np.abs(x) >= 2.0 ** -6
    rel = (err[big] / np.abs(x[big])).max()
    assert 2.0 ** -9 < rel <= 2.0 ** -8


def test_three_terms_hold_every_f16_value():
    x = _all("f16")
    err = np.abs(_split(x, 3) - x)
    assert err[np.abs(x) >= 2.0 ** -7].max() == 0
    assert err.max() <= 2.0 ** -18
