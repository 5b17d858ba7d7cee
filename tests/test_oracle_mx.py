"""Pins for the oracle's MXFP8 quantiser and blocked scale layout (oracle/mx.py).

The scale rule (shared exponent X = floor(log2 amax) - 8, E8M0 code X + 127)
and the e4m3 element codes are checked against values worked out by hand from
the definitions; the blocked layout against a second implementation built from
reshapes and transposes, hand-worked byte positions (tests/golden), and its
invariants."""
import json
import os

import numpy as np
import pytest

from oracle import mx as X
from oracle.formats import e4m3_decode

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_blocked_small.json")


def _run(vals):
    v = np.zeros((1, 32), dtype=np.float32)
    v[0, :len(vals)] = vals
    return X.mx_quantize(v)


def test_scale_codes_from_the_definition():
    # amax 1 -> X = 0 - 8; amax 500 -> floor(log2 500) = 8 -> X = 0
    assert _run([1.0])[1][0, 0] == 127 - 8
    assert _run([500.0, -3.0])[1][0, 0] == 127
    assert _run([-3.0 * 2.0 ** 100])[1][0, 0] == 127 + 93
    assert _run([1.5 * 2.0 ** 127])[1][0, 0] == 127 + 119
    assert _run([0.0, -0.0])[1][0, 0] == 0                     # all zero: X = -127
    assert _run([2.0 ** -130])[1][0, 0] == 0                   # below the range: clamped to X = -127
    assert _run([np.nextafter(np.float32(2.0), np.float32(0))])[1][0, 0] == 127 - 8  # just below 2: floor is 0


def test_element_codes_from_the_definition():
    codes, s = _run([1.0, 0.75, -0.5, 2.0 ** -10, 0.0, -0.0])
    # scale 2^-8: 1 -> 256 (exp field 15), 0.75 -> 192 = 1.5 * 2^7, -0.5 -> -128,
    # 2^-10 -> 2^-2 (exp field 5), zeros keep their sign
    assert codes[0, :6].tolist() == [0x78, 0x74, 0xF0, 0x28, 0x00, 0x80]
    codes, s = _run([500.0, 450.0, -464.0, 448.0, 1.0])
    assert s[0, 0] == 127
    assert codes[0, :5].tolist() == [0x7E, 0x7E, 0xFE, 0x7E, 0x38]  # saturate to +-448
    codes, s = _run([3.0 * 2.0 ** 100])
    assert codes[0, 0] == 0x7C  # 3 * 2^100 / 2^93 = 384 = 1.5 * 2^8
    codes, _ = _run([2.0 ** -130])
    assert codes[0, 0] == 0x20  # 2^-130 / 2^-127 = 2^-3 (exp field 4)


def test_runs_are_independent_and_round_trip_within_half_an_e4m3_step():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal((7, 96)) * np.exp2(rng.integers(-20, 20, size=(7, 96)))).astype(np.float32)
    codes, s = X.mx_quantize(v)
    assert s.shape == (7, 3)
    for r in range(7):
        for b in range(3):
            c1, s1 = X.mx_quantize(v[r:r + 1, 32 * b:32 * b + 32])
            assert np.array_equal(c1[0], codes[r, 32 * b:32 * b + 32]) and s1[0, 0] == s[r, b]
    back = X.mx_dequantize(codes, s)
    scale = X.e8m0_value(np.repeat(s, 32, axis=1))
    big = np.abs(v) >= scale * 2.0 ** -6       # e4m3 normal range after scaling
    unsat = np.abs(v) <= scale * 448.0
    m = big & unsat
    assert np.all(np.abs(back[m] - v[m]) <= np.abs(v[m]) * 2.0 ** -4 * (1 + 1e-12))
    assert np.all(np.abs(back[~unsat]) == scale[~unsat] * 448.0)  # saturated elements
    assert np.array_equal(e4m3_decode(codes) == 0, back == 0)


def test_blocked_layout_two_implementations_agree():
    rng = np.random.default_rng(1)
    for n, c in [(1, 1), (128, 4), (130, 5), (257, 64), (31, 24), (384, 160)]:
        sc = rng.integers(1, 255, size=(n, c)).astype(np.uint8)
        a = X.to_blocked(sc)
        b = X.to_blocked_by_reshape(sc)
        assert a.shape == b.shape == (-(-n // 128) * 128, -(-c // 4) * 4)
        assert np.array_equal(a, b)


def test_blocked_layout_hand_worked_positions_and_padding():
    g = json.load(open(GOLDEN))["single"]
    n, c = g["rows"], g["cols"]
    sc = (np.arange(n * c).reshape(n, c) % 251 + 1).astype(np.uint8)  # nonzero everywhere
    out = X.to_blocked(sc)
    assert out.shape == (g["padded_rows"], g["padded_cols"])
    flat = out.reshape(-1)
    for r, col, pos in g["positions"]:
        assert flat[pos] == sc[r, col], (r, col, pos)
    for pos in g["zero_positions"]:
        assert flat[pos] == 0
    # invariants: the valid scales map one-to-one onto the nonzero bytes, the rest is padding
    assert np.count_nonzero(flat) == n * c
    assert sorted(flat[flat != 0].tolist()) == sorted(sc.reshape(-1).tolist())


def test_per_group_starts_and_placement():
    g = json.load(open(GOLDEN))["groups"]
    rows, cols = g["rows"], g["cols"]
    off = np.concatenate([[0], np.cumsum(rows)])
    sc = (np.arange(off[-1] * cols).reshape(-1, cols) % 251 + 1).astype(np.uint8)
    out, starts = X.per_group_blocked(sc, off)
    assert starts.tolist() == g["starts"]
    flat = out.reshape(-1)
    for r, col, pos in g["positions"]:
        assert flat[pos] == sc[r, col], (r, col, pos)
    for gi in range(len(rows)):  # each group equals its own conversion
        blk = X.to_blocked(sc[off[gi]:off[gi + 1]]) if rows[gi] else np.zeros((0, 8), np.uint8)
        assert np.array_equal(out[starts[gi]:starts[gi + 1]], blk)
