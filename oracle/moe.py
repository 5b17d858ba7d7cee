"""Routed MoE FFN forward, written out plainly (oracle side; test infrastructure).

What is computed, step by step (the pipeline of "perf: add small-batch route
MMA for MoE", Motivation, and of "Port necessary FBGEMM MoE kernels",
index_shuffling + scatter_add_dense_tokens):

  1. route    per token t: the k experts with the largest router score, ordered
              by (score descending, expert id ascending) - ties go to the lower
              expert id, and -0.0 ties +0.0; combine weights w[t, j] = softmax
              over the k selected scores.
  2. shuffle  counts[e] = number of routes r = t*k + j with ids[t, j] == e;
              offsets = exclusive prefix sum of counts (length E+1); perm = the
              stable sort of the routes by expert (sorted position -> route
              r); inv[perm[p]] = p.
  3. tiles    for each expert with c_e > 0, ceil(c_e / BM) tiles (e, row0, nrows)
              covering its segment of sorted positions (the GEMM task map).
  4. FFN      per route r (token t, expert e):
                 [g | u] = W1[e] x_t       (W1[e] rows 0..I-1 = gate, I..2I-1 = up)
                 a = silu(g) * u           (silu(g) = g / (1 + exp(-g)))
                 h = a rounded to the Down GEMM's input type
                 o_r = W2[e] h
  5. combine  y[t] = sum_j w[t, j] * o_(t*k+j), rounded to bf16 once.

Quantisation modes (Summary of the route-MMA page: per-tensor and 128x128
blockwise FP8; the page does not define the rounding, so the plainest reading
is used, and the same rule serves every quantised tensor):

  bf16         h = bf16(a).
  fp8 tensor   x is quantised with one dynamic scale s_x = amax|x| / 448 over
               the whole [T, H] input, q_x = e4m3(x / s_x); weights arrive as
               e4m3 codes with one fp32 scale per expert matrix (W1[e], W2[e]);
               g = (s_x * s_w1[e]) * sum_h q_x q_w1, likewise u; h is quantised
               with one dynamic scale over all R x I values of a; o = (s_h *
               s_w2[e]) * sum_i q_h q_w2.
  mxfp8        OCP MX with e4m3 elements (the format of "[mxfp8 moe training]
               add per group blocked scale kernels", Summary; rule in oracle/mx.py):
               x and h are quantised per run of 32 consecutive values along the
               contraction dimension with a power-of-two (E8M0) scale; weights
               arrive as e4m3 codes with E8M0 scales [E, rows, K/32]; every
               operand is the exact product code * 2^X, so the GEMMs contract
               the dequantised values.
  fp8 block    x scales per (token, 128-column group); weight scales per
               128 x 128 block; g_i = sum_G s_x[t, G] s_w1[e, i//128, G] *
               sum_{h in G} q_x q_w1 (the up row I+i uses block row
               (I+i)//128); h scales per (route, 128-column group of I); o_c =
               sum_G s_h[r, G] s_w2[e, c//128, G] * sum_{i in G} q_h q_w2.

Every scale is s = amax / 448 in fp32 (s = 1 when amax == 0); q = e4m3(v / s)
with an fp32 IEEE division and round-to-nearest-even, saturating.  Dot products
and sums are accumulated in fp64; a is rounded to fp32 before it is quantised,
so the quantisation decision is taken in fp32 as the kernels take it.

Pins (tests/test_oracle_route_shuffle.py, tests/test_oracle_forward.py): brute
force top-k on tiny inputs, tie and signed-zero cases, k = E and k = 1 closed
forms, the two-expert softmax = logistic sigmoid closed form; two independent
shuffle implementations (stable sort and counting placement) plus the shuffle
and tile-map invariants; the identity-expert closed form of the FFN in all
three modes; the E = 1, k = 1 dense SwiGLU MLP against torch CPU; a brute-force
dense sum over all experts with zero gates for unselected ones.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from .formats import (
    E4M3_MAX,
    bf16_round,
    e4m3_decode,
    e4m3_encode,
    f32_from_bf16_bits,
)
from .mx import mx_dequantize, mx_quantize

BF16 = "bf16"
FP8_TENSOR = "fp8_tensor"
FP8_BLOCK = "fp8_block"
MXFP8 = "mxfp8"
GROUP = 128  # 128-wide scale groups of the blockwise mode


# ----------------------------------------------------------------------------- 1. route
def route(scores: np.ndarray, k: int):
    """Top-k routing.  scores fp32 [T, E] -> ids int32 [T, k], w fp32 [T, k].

    Order: score descending, expert id ascending among equal scores (IEEE
    comparison, so -0.0 == +0.0 and falls to the id).  A stable sort of the
    negated scores gives exactly that order.  Softmax over the k selected
    scores: m = the largest selected score, e_j = exp(s_j - m), w_j = e_j / sum e."""
    s = np.asarray(scores, dtype=np.float32)
    T, E = s.shape
    assert 1 <= k <= E
    order = np.argsort(-s, axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(s, ids, axis=1).astype(np.float64)
    m = sel[:, :1]
    e = np.exp(sel - m)
    w = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


# ----------------------------------------------------------------------------- 2. shuffle
def shuffle(ids: np.ndarray, E: int):
    """Index shuffling.  ids int32 [T, k] (or flat [R]) -> counts [E],
    offsets [E+1], perm [R] (sorted position -> route id r = t*k + j), inv [R]."""
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return counts, offsets, perm, inv


def shuffle_by_counting(ids: np.ndarray, E: int):
    """The same shuffle by counting placement: walk the routes in order and drop
    each into the next free slot of its expert's segment.  Used only as the
    independent second implementation that pins ``shuffle``."""
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    counts = [0] * E
    for e in flat:
        counts[e] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    nxt = offsets[:E]
    nxt = list(nxt)
    perm = [0] * len(flat)
    for r, e in enumerate(flat):
        perm[nxt[e]] = r
        nxt[e] += 1
    inv = [0] * len(flat)
    for p, r in enumerate(perm):
        inv[r] = p
    as32 = lambda v: np.asarray(v, dtype=np.int32)
    return as32(counts), as32(offsets), as32(perm), as32(inv)


# ----------------------------------------------------------------------------- 3. tile map
def tile_map(counts: np.ndarray, BM: int) -> np.ndarray:
    """GEMM task map: for each expert in id order with c_e > 0, ceil(c_e / BM)
    row tiles (e, row0, nrows) over its segment of sorted positions.  Returns
    int32 [ntiles, 3]; experts without routes contribute no tile."""
    tiles = []
    row = 0
    for e, c in enumerate(np.asarray(counts).tolist()):
        for j in range(0, c, BM):
            tiles.append((e, row + j, min(BM, c - j)))
        row += c
    return np.asarray(tiles, dtype=np.int32).reshape(-1, 3)


# ----------------------------------------------------------------------------- quantisers
def scale_of(amax: np.ndarray) -> np.ndarray:
    """s = amax / 448 in fp32; s = 1 where amax == 0."""
    a = np.asarray(amax, dtype=np.float32)
    s = a / np.float32(E4M3_MAX)
    return np.where(a == 0, np.float32(1.0), s).astype(np.float32)


def quant_per_tensor(v: np.ndarray):
    """One dynamic scale over the whole tensor.  -> (codes uint8, scale fp32 scalar)."""
    v = np.asarray(v, dtype=np.float32)
    s = scale_of(np.abs(v).max() if v.size else np.float32(0))
    return e4m3_encode(v / s), np.float32(s)


def quant_per_group(v: np.ndarray, group: int = GROUP):
    """One dynamic scale per (row, group of ``group`` columns); the last group
    covers the remaining columns.  v fp32 [rows, cols] -> (codes uint8 [rows,
    cols], scales fp32 [rows, ceil(cols / group)])."""
    v = np.asarray(v, dtype=np.float32)
    rows, cols = v.shape
    ng = -(-cols // group)
    codes = np.empty((rows, cols), dtype=np.uint8)
    scales = np.empty((rows, ng), dtype=np.float32)
    for G in range(ng):
        blk = v[:, G * group:(G + 1) * group]
        s = scale_of(np.abs(blk).max(axis=1))
        scales[:, G] = s
        codes[:, G * group:(G + 1) * group] = e4m3_encode(blk / s[:, None])
    return codes, scales


# ----------------------------------------------------------------------------- 4.-5. forward
def silu_times(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """SwiGLU activation a = silu(g) * u = g / (1 + exp(-g)) * u (fp64)."""
    return g / (1.0 + np.exp(-g)) * u


def _decode_input(arr, quant):
    """x / weights: bf16 arrive as uint16 bit patterns, FP8 weights as uint8 codes."""
    if arr.dtype == np.uint16:
        return f32_from_bf16_bits(arr)
    if arr.dtype == np.uint8:
        return e4m3_decode(arr)
    return np.asarray(arr, dtype=np.float32)


def forward(
    x_bits: np.ndarray,
    scores: np.ndarray,
    w1: np.ndarray,
    w2: np.ndarray,
    w1_scale: Optional[np.ndarray],
    w2_scale: Optional[np.ndarray],
    k: int,
    quant: str,
    tokens: Optional[np.ndarray] = None,
    shared: Optional[Dict[str, np.ndarray]] = None,
    y_fp32: bool = False,
) -> Dict[str, np.ndarray]:
    """The full forward.

    x_bits   uint16 [T, H]        bf16 bit patterns of x
    scores   fp32   [T, E]
    w1       [E, 2I, H]           bf16 bits (uint16) or e4m3 codes (uint8)
    w2       [E, H, I]            same
    w1_scale None | fp32 [E] | fp32 [E, ceil(2I/128), ceil(H/128)] | E8M0 uint8 [E, 2I, H/32] (mxfp8)
    w2_scale None | fp32 [E] | fp32 [E, ceil(H/128), ceil(I/128)] | E8M0 uint8 [E, H, I/32] (mxfp8)
    tokens   optional subset of token indices: y is computed only for those
             (all routes are still computed when a per-tensor scale of h needs
             them).
    shared   optional shared experts (the "shared output" of the route-MMA
             page's Summary): {"w1": [S, 2I, H], "w2": [S, H, I], "w1_scale",
             "w2_scale"} in the routed experts' formats.  Every token passes
             through every shared expert with weight 1.  Their rows are more
             rows of the same intermediate tensor: x is quantised once for
             both, and the per-tensor scale of h spans routed and shared rows.
             y[t] = sum_j w[t, j] o_(t*k+j) + sum_s o_shared(s, t), summed in
             that order, rounded once.
    y_fp32   return y unrounded (fp32 of the sum): the partial output of one
             slice of a tensor-parallel split of I, to be summed across the
             slices and rounded once by the caller.

    Returns a dict with ids, w, counts, offsets, perm, inv, a (fp32 [R, I] for
    the computed routes, NaN elsewhere; with shared experts [R + S*T, I], row
    R + s*T + t for shared expert s and token t), y (fp32 holding bf16
    values unless y_fp32, [T, H] or [len(tokens), H])."""
    x = f32_from_bf16_bits(x_bits)
    T, H = x.shape
    E, twoI, _ = w1.shape
    I = twoI // 2
    R = T * k
    ids, w = route(scores, k)
    counts, offsets, perm, inv = shuffle(ids, E)
    ids_flat = ids.reshape(-1)
    S = 0 if shared is None else int(shared["w1"].shape[0])
    if S:
        # shared expert s is expert E + s of an extended expert set, and its rows
        # R + s*T + t are extra routes that every token takes
        w1 = np.concatenate([w1, shared["w1"]], axis=0)
        w2 = np.concatenate([w2, shared["w2"]], axis=0)
        if quant != BF16:
            w1_scale = np.concatenate([w1_scale, shared["w1_scale"]], axis=0)
            w2_scale = np.concatenate([w2_scale, shared["w2_scale"]], axis=0)
        seg_of = [perm[offsets[e]:offsets[e + 1]] for e in range(E)]
        seg_of += [R + s * T + np.arange(T) for s in range(S)]
    else:
        seg_of = [perm[offsets[e]:offsets[e + 1]] for e in range(E)]
    RS = R + S * T

    def token_of(rows):
        return np.where(rows < R, rows // k, (rows - R) % T)

    if tokens is None:
        tokens = np.arange(T)
    tokens = np.asarray(tokens, dtype=np.int64)
    need = np.zeros(RS, dtype=bool)
    for t in tokens:
        need[t * k:(t + 1) * k] = True
        need[R + t:RS:T] = True
    gate_up_need = np.ones(RS, dtype=bool) if quant == FP8_TENSOR else need

    # activation quantisation of x
    if quant == BF16:
        xv = x.astype(np.float64)
    elif quant == FP8_TENSOR:
        xq, sx = quant_per_tensor(x)
        xv = e4m3_decode(xq).astype(np.float64)
    elif quant == FP8_BLOCK:
        xq, sxg = quant_per_group(x)
        xv = e4m3_decode(xq).astype(np.float64)
    elif quant == MXFP8:
        xq, sxm = mx_quantize(x)
        xv = mx_dequantize(xq, sxm)
    else:
        raise ValueError(quant)

    a = np.full((RS, I), np.nan, dtype=np.float32)
    # Gate/Up per expert over its routes in sorted order (perm order), then the
    # shared experts over every token
    for e in range(E + S):
        seg = seg_of[e]
        seg = seg[gate_up_need[seg]]
        if seg.size == 0:
            continue
        tok = token_of(seg)
        if quant == MXFP8:
            W1e = mx_dequantize(w1[e], w1_scale[e])
        else:
            W1e = _decode_input(w1[e], quant).astype(np.float64)
        Xe = xv[tok]
        if quant in (BF16, MXFP8):
            g = Xe @ W1e[:I].T
            u = Xe @ W1e[I:].T
        elif quant == FP8_TENSOR:
            sc = np.float64(sx) * np.float64(w1_scale[e])
            g = sc * (Xe @ W1e[:I].T)
            u = sc * (Xe @ W1e[I:].T)
        else:
            gu = np.zeros((seg.size, 2 * I), dtype=np.float64)
            for G in range(-(-H // GROUP)):
                hs = slice(G * GROUP, (G + 1) * GROUP)
                part = Xe[:, hs] @ W1e[:, hs].T  # [n, 2I]
                rowblk = np.arange(2 * I) // GROUP
                sw = w1_scale[e][rowblk, G].astype(np.float64)  # [2I]
                gu += sxg[tok, G].astype(np.float64)[:, None] * sw[None, :] * part
            g, u = gu[:, :I], gu[:, I:]
        a[seg] = silu_times(g, u).astype(np.float32)

    # quantisation of h (the Down GEMM's input)
    hv = np.zeros((RS, I), dtype=np.float64)
    if quant == BF16:
        hv[need] = bf16_round(a[need])
    elif quant == FP8_TENSOR:
        hq, sh = quant_per_tensor(a)
        hv = e4m3_decode(hq).astype(np.float64)
    elif quant == MXFP8:
        hq, shm = mx_quantize(a[need])
        hv[need] = mx_dequantize(hq, shm)
    else:
        shg = np.zeros((RS, -(-I // GROUP)), dtype=np.float32)
        hq, shg_need = quant_per_group(a[need])
        hv[need] = e4m3_decode(hq)
        shg[need] = shg_need

    # Down per expert (and shared expert), o in route order
    o = np.zeros((RS, H), dtype=np.float64)
    for e in range(E + S):
        seg = seg_of[e]
        seg = seg[need[seg]]
        if seg.size == 0:
            continue
        if quant == MXFP8:
            W2e = mx_dequantize(w2[e], w2_scale[e])
        else:
            W2e = _decode_input(w2[e], quant).astype(np.float64)
        He = hv[seg]
        if quant in (BF16, MXFP8):
            o[seg] = He @ W2e.T
        elif quant == FP8_TENSOR:
            o[seg] = (np.float64(sh) * np.float64(w2_scale[e])) * (He @ W2e.T)
        else:
            acc = np.zeros((seg.size, H), dtype=np.float64)
            for G in range(-(-I // GROUP)):
                cs = slice(G * GROUP, (G + 1) * GROUP)
                part = He[:, cs] @ W2e[:, cs].T  # [n, H]
                sw = w2_scale[e][np.arange(H) // GROUP, G].astype(np.float64)  # [H]
                acc += shg[seg, G].astype(np.float64)[:, None] * sw[None, :] * part
            o[seg] = acc

    # combine: y[t] = bf16(sum_j w[t, j] o[t*k + j] + sum_s o_shared(s, t)),
    # j ascending, then s ascending
    y = np.empty((tokens.size, H), dtype=np.float32)
    for n, t in enumerate(tokens):
        acc = np.zeros(H, dtype=np.float64)
        for j in range(k):
            acc += np.float64(w[t, j]) * o[t * k + j]
        for s_ in range(S):
            acc += o[R + s_ * T + t]
        y[n] = acc.astype(np.float32) if y_fp32 else bf16_round(acc.astype(np.float32))

    return {
        "ids": ids,
        "w": w,
        "counts": counts,
        "offsets": offsets,
        "perm": perm,
        "inv": inv,
        "ids_flat": ids_flat,
        "a": a,
        "y": y,
        "tokens": tokens,
    }
