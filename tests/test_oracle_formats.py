"""Pins for the oracle's storage formats (OCP E4M3 and bfloat16).

The oracle's codecs are written from the formats' bit definitions; these tests
tie them to facts that do not come from the oracle itself: exhaustive
round-trips over every E4M3 code, the format's textbook values, exact
midpoints (round-to-nearest-even), saturation, and torch's own casts.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _finite_codes():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_e4m3_textbook_values():
    # OCP 8-bit floating point, E4M3: bias 7, 3 mantissa bits, max 448,
    # smallest normal 2^-6, smallest subnormal 2^-9, no infinities.
    table = {0x00: 0.0, 0x80: -0.0, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0,
             0x08: 2.0**-6, 0x01: 2.0**-9, 0x07: 7 * 2.0**-9, 0x77: 240.0, 0x30: 0.5}
    for code, val in table.items():
        got = oracle.e4m3_decode([code])[0]
        assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)
    assert np.isnan(oracle.e4m3_decode([0x7F])[0]) and np.isnan(oracle.e4m3_decode([0xFF])[0])


def test_e4m3_roundtrip_every_code():
    codes = np.array(_finite_codes(), dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    back = oracle.e4m3_encode(vals)
    assert np.array_equal(back, codes)


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes.numpy())
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[fin], ref[fin])


def test_e4m3_midpoints_round_to_even():
    pos = [c for c in _finite_codes() if c < 0x7E]  # adjacent pairs (c, c+1) up to 448
    lo = oracle.e4m3_decode(np.array(pos, dtype=np.uint8))
    hi = oracle.e4m3_decode(np.array(pos, dtype=np.uint8) + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)  # exact in binary32
    got = oracle.e4m3_encode(mid)
    want = np.where(np.array(pos) % 2 == 0, np.array(pos), np.array(pos) + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    # just off the midpoint goes to the nearer neighbour
    up = np.nextafter(mid, np.float32(np.inf))
    dn = np.nextafter(mid, np.float32(-np.inf))
    assert np.array_equal(oracle.e4m3_encode(up), (np.array(pos) + 1).astype(np.uint8))
    assert np.array_equal(oracle.e4m3_encode(dn), np.array(pos, dtype=np.uint8))
    # negative side mirrors
    assert np.array_equal(oracle.e4m3_encode(-mid), want | 0x80)


def test_e4m3_saturates_and_nan():
    big = np.array([448.0, 449.0, 464.0, 464.1, 480.0, 1e6, np.inf], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    assert oracle.e4m3_encode([np.nan])[0] & 0x7F == 0x7F
    # underflow: below half the smallest subnormal rounds to (signed) zero
    tiny = np.array([2.0**-11, 2.0**-10], dtype=np.float32)  # 2^-10 is a tie -> even (0)
    assert np.all(oracle.e4m3_encode(tiny) == 0x00)
    assert np.all(oracle.e4m3_encode(-tiny) == 0x80)
    assert oracle.e4m3_encode([1.5 * 2.0**-10])[0] == 0x01


@pytest.mark.parametrize("scale_exp", [-12, -8, -3, 0, 3, 6, 8])
def test_e4m3_encode_matches_torch_in_range(scale_exp):
    g = torch.Generator().manual_seed(100 + scale_exp)
    x = (torch.randn(50000, generator=g) * 2.0**scale_exp).clamp(-464.0, 464.0)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.numpy())
    assert np.array_equal(got, ref)


def test_bf16_matches_torch():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(100000, generator=g) * torch.exp(torch.randn(100000, generator=g) * 10)
    # add exact ties: values whose low 16 bits are 0x8000
    ties = (torch.randint(0, 2**15, (1000,), generator=g, dtype=torch.int32) << 16) | 0x8000
    x = torch.cat([x, ties.view(torch.float32)])
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_encode(x.numpy())
    fin = np.isfinite(x.numpy())
    assert np.array_equal(got[fin], ref[fin])
    back = oracle.bf16_decode(ref)
    assert np.array_equal(back, x.to(torch.bfloat16).to(torch.float64).numpy(), equal_nan=True)
