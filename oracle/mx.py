"""MXFP8 quantisation and the per-group blocked scale layout (oracle side; test
infrastructure only, like the rest of this package).

Source: "[mxfp8 moe training] add per group blocked scale kernels" (pytorch/ao
PR 2886), Summary: MX scales of 2D input activations, grouped by expert, are
converted into the blocked, swizzled layout per group, with the start row of
each group in the block-padded output computed on the device.  The page names
the formats but defines neither the MX quantisation nor the blocked layout;
the plainest readings are taken:

MXFP8 (the OCP Microscaling format with E4M3 elements): every run of 32
consecutive values along a row (the GEMM's K dimension) shares one E8M0 scale
2^X, an 8-bit biased exponent (code = X + 127; code 255 is NaN and never
produced).  X = floor(log2(amax)) - 8, where 8 is the exponent of the largest
e4m3 power of two (448 = 1.75 * 2^8), clamped to [-127, 127]; an all-zero run
takes X = -127.  Elements are e4m3(v / 2^X), rounded to nearest even and
saturated to +-448 (amax / 2^X lies in [256, 512), so the run's largest values
may saturate).

Blocked layout: a scale matrix [rows, cols] (one byte per scale) is padded with
zeros to a multiple of 128 rows and 4 columns and cut into 128 x 4 blocks,
stored block row by block row, each block as 512 contiguous bytes in which the
scale of (row r, column c) of the block sits at byte (r mod 32) * 16 +
(r div 32) * 4 + c: 32 lines of 16 bytes, line i holding rows i, i+32, i+64,
i+96 of the block, four columns each.  Per group: each group's rows are
converted on their own, padded to a multiple of 128 rows, and the groups'
padded blocks follow one another; group g starts at padded row
sum_{h<g} ceil(n_h / 128) * 128.

Pins (tests/test_oracle_mx.py): scale exponents and codes worked by hand from the
definition above; the e4m3 element rule reduces to the oracle's pinned e4m3
encoder on exact powers of two; the blocked layout against a second, independent
implementation (reshapes and transposes instead of the index formula), against
hand-worked byte positions (tests/golden/mx_blocked_small.json) and against its
invariants (a bijection of the valid scales onto the non-padding bytes, zero
padding, 512-byte blocks).
"""
from __future__ import annotations

import numpy as np

from .formats import e4m3_decode, e4m3_encode

MX_BLOCK = 32       # values per shared scale
E4M3_EMAX = 8       # exponent of the largest e4m3 power of two (448 = 1.75 * 2^8)
BLOCK_ROWS = 128    # rows of one blocked-layout block
BLOCK_COLS = 4      # scale columns of one blocked-layout block


def floor_log2(a: np.ndarray) -> np.ndarray:
    """floor(log2(a)) of positive finite fp32 values, exactly (from the binary
    exponent: a = f * 2^e with f in [0.5, 1), so floor(log2 a) = e - 1)."""
    _, e = np.frexp(np.asarray(a, dtype=np.float64))
    return e.astype(np.int64) - 1


def mx_exponent(amax: np.ndarray) -> np.ndarray:
    """The shared exponent X of a run with the given amax (fp32 >= 0)."""
    a = np.asarray(amax, dtype=np.float32)
    x = np.full(a.shape, -127, dtype=np.int64)
    pos = a > 0
    x[pos] = floor_log2(a[pos]) - E4M3_EMAX
    return np.clip(x, -127, 127)


def e8m0_value(codes: np.ndarray) -> np.ndarray:
    """E8M0 scale codes -> 2^(code - 127) in fp64 (exact)."""
    return np.ldexp(1.0, np.asarray(codes, dtype=np.int64) - 127)


def mx_quantize(v: np.ndarray):
    """v fp32 [rows, cols] (cols a multiple of 32) -> (e4m3 codes uint8 [rows,
    cols], E8M0 scale codes uint8 [rows, cols / 32])."""
    v = np.asarray(v, dtype=np.float32)
    rows, cols = v.shape
    assert cols % MX_BLOCK == 0
    runs = v.reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    X = mx_exponent(np.abs(runs).max(axis=2))
    scaled = (runs.astype(np.float64) / np.ldexp(1.0, X)[:, :, None]).astype(np.float32)
    codes = e4m3_encode(scaled).reshape(rows, cols)
    return codes, (X + 127).astype(np.uint8)


def mx_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Inverse map (exact in fp64): value = e4m3(code) * 2^(scale code - 127)."""
    c = np.asarray(codes)
    rows, cols = c.shape
    v = e4m3_decode(c).astype(np.float64).reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    return (v * e8m0_value(scales)[:, :, None]).reshape(rows, cols)


def padded_cols(cols: int) -> int:
    return -(-cols // BLOCK_COLS) * BLOCK_COLS


def blocked_group_starts(group_rows) -> np.ndarray:
    """Start row of each group in the block-padded output, and the total rows
    (entry G): start[g + 1] = start[g] + ceil(n_g / 128) * 128."""
    n = np.asarray(group_rows, dtype=np.int64)
    starts = np.zeros(n.size + 1, dtype=np.int64)
    starts[1:] = np.cumsum(-(-n // BLOCK_ROWS) * BLOCK_ROWS)
    return starts


def to_blocked(sc: np.ndarray) -> np.ndarray:
    """One group's scales [n, cols] -> its blocked bytes [ceil(n/128)*128, padded_cols]
    (row-major view of the flat block sequence), by the index formula."""
    sc = np.asarray(sc, dtype=np.uint8)
    n, cols = sc.shape
    prow = -(-n // BLOCK_ROWS) * BLOCK_ROWS
    pcol = padded_cols(cols)
    ncb = pcol // BLOCK_COLS
    out = np.zeros(prow * pcol, dtype=np.uint8)
    for r in range(n):
        rb, rr = divmod(r, BLOCK_ROWS)
        for c in range(cols):
            cb, cc = divmod(c, BLOCK_COLS)
            out[(rb * ncb + cb) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + cc] = sc[r, c]
    return out.reshape(prow, pcol)


def to_blocked_by_reshape(sc: np.ndarray) -> np.ndarray:
    """The same layout by reshapes and transposes: pad, cut into 128 x 4 blocks
    (block rows outer), split each block's 128 rows into 4 groups of 32 and
    interleave them so that line i holds rows i, i+32, i+64, i+96.  Used only as
    the independent second implementation that pins ``to_blocked``."""
    sc = np.asarray(sc, dtype=np.uint8)
    n, cols = sc.shape
    prow = -(-n // BLOCK_ROWS) * BLOCK_ROWS
    pcol = padded_cols(cols)
    pad = np.zeros((prow, pcol), dtype=np.uint8)
    pad[:n, :cols] = sc
    blocks = pad.reshape(prow // 128, 128, pcol // 4, 4).transpose(0, 2, 1, 3)  # [rb, cb, 128, 4]
    lines = blocks.reshape(-1, 4, 32, 4).transpose(0, 2, 1, 3)                  # [blk, 32, 4 (row group), 4]
    return lines.reshape(prow, pcol)


def per_group_blocked(sc: np.ndarray, group_offsets) -> tuple:
    """Scales [M, cols] whose rows are grouped (group g = rows [off[g],
    off[g+1])) -> (blocked output [starts[G], padded_cols], starts [G+1])."""
    sc = np.asarray(sc, dtype=np.uint8)
    off = np.asarray(group_offsets, dtype=np.int64)
    starts = blocked_group_starts(np.diff(off))
    out = np.zeros((int(starts[-1]), padded_cols(sc.shape[1])), dtype=np.uint8)
    for g in range(off.size - 1):
        if off[g + 1] > off[g]:
            out[starts[g]:starts[g + 1]] = to_blocked(sc[off[g]:off[g + 1]])
    return out, starts
