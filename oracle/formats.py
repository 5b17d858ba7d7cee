"""Number formats used by the routed MoE forward (oracle side; test infrastructure).

bf16: IEEE-754 binary32 with the low 16 fraction bits dropped.  Rounding from
fp32 is round-to-nearest, ties-to-even (the IEEE default), applied to the bit
pattern.  Inputs are finite (non-finite router scores and activations are
outside the contract).

e4m3: the OCP 8-bit floating point format E4M3 ("FN" variant): 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
subnormals m/8 * 2^-6; there is no infinity; S.1111.111 is NaN; the largest
finite magnitude is 1.75 * 2^8 = 448.  Conversion from fp32 rounds to nearest,
ties to even, and saturates to +-448 (the "satfinite" conversion used by the
FP8 quantisation of "perf: add small-batch route MMA for MoE", Summary: per-
tensor and 128x128 blockwise FP8).

Pins (tests/test_oracle_formats.py): every bf16 pattern round-trips; fp32 -> bf16
agrees with torch's conversion on random and midpoint values; the e4m3 table
matches values fixed by the format definition; every e4m3 code round-trips;
every midpoint between neighbouring codes rounds to the even code; in-range
values agree with torch's float8_e4m3fn conversion; out-of-range values
saturate.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


# ----------------------------------------------------------------------------- bf16
def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16
    return (u & 0xFFFF).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 value (ties to even); returns fp32."""
    return f32_from_bf16_bits(bf16_bits_from_f32(np.asarray(a, dtype=np.float32)))


# ----------------------------------------------------------------------------- e4m3
def _e4m3_table() -> np.ndarray:
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        man = code & 0x7
        if exp_field == 0xF and man == 0x7:
            vals[code] = np.nan
        elif exp_field == 0:
            vals[code] = sign * (man / 8.0) * 2.0 ** (1 - 7)
        else:
            vals[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp_field - 7)
    return vals.astype(np.float32)


E4M3_VALUES = _e4m3_table()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """e4m3 codes (uint8) -> fp32 values (exact)."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """fp32 values -> e4m3 codes: round to nearest, ties to even, saturating to
    +-448.  The sign of the input is kept (a negative value that rounds to zero
    gives the negative-zero code 0x80).

    Derivation: for |v| >= 2^-6 (the smallest normal), with 2^e <= |v| < 2^(e+1)
    the representable neighbours are spaced 2^(e-3) apart, so the significand
    count n = |v| / 2^(e-3) lies in [8, 16) and is rounded to an integer with
    ties to even; n = 16 carries into the next binade.  Below 2^-6 the spacing
    is the subnormal quantum 2^-9.  Every division here is by a power of two and
    therefore exact in fp64."""
    v32 = np.asarray(v, dtype=np.float32)
    a = np.abs(v32).astype(np.float64)
    neg = np.signbit(v32)
    code = np.zeros(a.shape, dtype=np.int64)

    sub = a < 2.0 ** -6
    n_sub = np.rint(a[sub] / 2.0 ** -9).astype(np.int64)  # 0..8; 8 == smallest normal
    code[sub] = n_sub

    nrm = ~sub
    an = a[nrm]
    _, ex = np.frexp(an)  # an = f * 2^ex, f in [0.5, 1)
    e = ex.astype(np.int64) - 1
    n = np.rint(an / np.ldexp(1.0, e - 3)).astype(np.int64)  # in [8, 16]
    carry = n == 16
    e = np.where(carry, e + 1, e)
    n = np.where(carry, 8, n)
    c = ((e + 7) << 3) | (n - 8)
    # saturation: anything beyond 448 (code 0x7E) clamps to 448
    c = np.where((e + 7 > 15) | (c > 0x7E), 0x7E, c)
    code[nrm] = c

    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """fp32 -> nearest e4m3 value (ties to even, saturating), returned as fp32."""
    return e4m3_decode(e4m3_encode(v))
