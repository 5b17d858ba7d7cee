"""Pins for the oracle's number formats (bf16 RNE, OCP e4m3 RNE-satfinite).

Each check is against something other than the oracle itself: values fixed by
the format definitions, exhaustive round-trips, exact midpoints, and torch's
own conversions (library routines) where they apply."""
import numpy as np
import pytest
import torch

from oracle import formats as F


def test_bf16_all_patterns_round_trip():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = F.f32_from_bf16_bits(bits)
    finite = np.isfinite(vals)
    back = F.bf16_bits_from_f32(vals[finite])
    assert np.array_equal(back, bits[finite])


def test_bf16_matches_torch_on_random_fp32():
    rng = np.random.default_rng(0)
    mant = rng.integers(0, 1 << 23, size=200_000, dtype=np.uint32)
    exp = rng.integers(1, 254, size=200_000, dtype=np.uint32)
    sign = rng.integers(0, 2, size=200_000, dtype=np.uint32)
    u = (sign << 31) | (exp << 23) | mant
    v = u.view(np.float32)
    ref = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = F.bf16_bits_from_f32(v)
    ok = np.isfinite(torch.from_numpy(v.copy()).to(torch.bfloat16).float().numpy())
    assert np.array_equal(got[ok], ref[ok])


def test_bf16_midpoints_tie_to_even():
    # the fp32 value exactly halfway between two neighbouring bf16 values
    rng = np.random.default_rng(1)
    lo = rng.integers(0x0080, 0x7F00, size=5000).astype(np.uint32)
    mid = ((lo << 16) | 0x8000).view(np.float32)
    got = F.bf16_bits_from_f32(mid).astype(np.uint32)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, expect)
    # one fp32 ulp either side goes to the nearer neighbour
    below = np.nextafter(mid, np.float32(0))
    above = np.nextafter(mid, np.float32(np.inf))
    assert np.array_equal(F.bf16_bits_from_f32(below).astype(np.uint32), lo)
    assert np.array_equal(F.bf16_bits_from_f32(above).astype(np.uint32), lo + 1)


def test_e4m3_table_values_from_definition():
    t = F.E4M3_VALUES
    assert t[0x00] == 0.0 and not np.signbit(t[0x00])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    assert t[0x01] == 2.0 ** -9  # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9  # largest subnormal
    assert t[0x08] == 2.0 ** -6  # smallest normal
    assert t[0x38] == 1.0
    assert t[0x40] == 2.0
    assert t[0x3C] == 1.5
    assert t[0x7E] == 448.0  # largest finite
    assert t[0xFE] == -448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    pos = t[:0x7F].astype(np.float64)
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F])


def test_e4m3_codes_round_trip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(F.e4m3_encode(F.e4m3_decode(codes)), codes)


def test_e4m3_midpoints_tie_to_even_and_neighbours():
    pos = F.E4M3_VALUES[:0x7F].astype(np.float64)
    for c in range(0x7E):
        lo, hi = pos[c], pos[c + 1]
        mid = np.float32((lo + hi) / 2)  # exact: neighbours differ by a power of two
        assert np.float64(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert F.e4m3_encode(np.array([mid]))[0] == even
        assert F.e4m3_encode(np.array([-mid]))[0] == (even | 0x80)
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(np.inf))
        assert F.e4m3_encode(np.array([below]))[0] == c
        assert F.e4m3_encode(np.array([above]))[0] == c + 1


def test_e4m3_saturates_and_matches_torch_in_range():
    sat = np.array([448.0, 449.0, 463.9, 464.0, 470.0, 1e6, 3e38], dtype=np.float32)
    assert np.all(F.e4m3_encode(sat) == 0x7E)
    assert np.all(F.e4m3_encode(-sat) == 0xFE)
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(100_000) * np.exp(rng.uniform(-12, 5.5, 100_000))).astype(np.float32)
    v = v[np.abs(v) < 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.e4m3_encode(v)
    assert np.array_equal(F.e4m3_decode(got), F.e4m3_decode(ref))


@pytest.mark.parametrize("v,code", [(2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (2.0 ** -11, 0x00),
                                    (-(2.0 ** -11), 0x80), (15 * 2.0 ** -10, 0x08)])
def test_e4m3_subnormal_rounding(v, code):
    assert F.e4m3_encode(np.array([v], dtype=np.float32))[0] == code
