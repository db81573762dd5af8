"""Pins of the oracle's number formats against library routines and closed forms.

The oracle decodes fp16 / bf16 / fp8-e4m3 bits to fp64 and encodes fp32 to
e4m3 with its own C code written from the format definitions.  Here each is
checked exhaustively against numpy / PyTorch conversions (independent library
code) and against values that follow from the definitions by hand.
"""
import numpy as np
import pytest
import torch

import oracle


def test_f16_exhaustive_vs_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zero preserved
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_bf16_exhaustive_vs_torch():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]       # S.1111.111 only
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x38, 1.0),
    (0x3C, 1.5), (0x40, 2.0), (0x7E, 448.0), (0x77, 240.0), (0xB8, -1.0), (0xFE, -448.0),
])
def test_e4m3_decode_closed_forms(code, value):
    # value = (-1)^s * 2^(e-7) * (1 + f/8) for e > 0, (-1)^s * f * 2^-9 for e = 0
    assert oracle.e4m3_to_f64(np.array([code], np.uint8))[0] == value


def test_e4m3_encode_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_e4m3_encode_midpoints_round_to_even():
    """Halfway between neighbouring codes the encoder must pick the code whose
    last fraction bit is 0 (round to nearest, ties to even)."""
    pos = np.arange(0x00, 0x7E, dtype=np.uint8)           # 0 .. 416 (next is 448)
    lo = oracle.e4m3_to_f64(pos)
    hi = oracle.e4m3_to_f64(pos + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)  # exact in fp32
    got = oracle.e4m3_encode(mid)
    want = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.e4m3_encode(-mid), want | 0x80)
    # one ulp of fp32 either side of a midpoint decides the direction
    up = np.nextafter(mid, np.float32(np.inf))
    dn = np.nextafter(mid, np.float32(0))
    assert np.array_equal(oracle.e4m3_encode(up), pos + 1)
    assert np.array_equal(oracle.e4m3_encode(dn[1:]), pos[1:])


def test_e4m3_encode_saturates_and_nan():
    x = np.array([448.0, 449.0, 463.9, 464.0, 1e6, np.inf, -500.0, -np.inf], np.float32)
    assert oracle.e4m3_encode(x).tolist() == [0x7E] * 6 + [0xFE] * 2
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_e4m3_encode_random_vs_torch():
    """PyTorch's fp32 -> float8_e4m3fn cast rounds to nearest even inside the
    finite range (it does not saturate, so compare only |x| <= 448)."""
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 100,
                        rng.standard_normal(20000).astype(np.float32) * 0.01,
                        (rng.random(5000) * 896 - 448).astype(np.float32)])
    x = x[np.abs(x) <= 448]
    got = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
