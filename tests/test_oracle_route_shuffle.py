"""Pins for the oracle's routing, index shuffling and tile map.

Routing is checked against a brute-force comparator sort, hand-worked goldens,
the k = E / k = 1 special cases and the two-expert closed form of the softmax
(the logistic function).  The shuffle is checked against an independent
counting-placement implementation, hand-worked goldens and its invariants."""
import functools
import json
import math
import os

import numpy as np
import pytest

from oracle import moe as M

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _brute_order(row):
    """Expert order by a comparator: larger score first, lower id on equal scores."""
    def cmp(i, j):
        if row[i] > row[j]:
            return -1
        if row[i] < row[j]:
            return 1
        return -1 if i < j else (1 if i > j else 0)
    return sorted(range(len(row)), key=functools.cmp_to_key(cmp))


@pytest.mark.parametrize("seed", range(20))
def test_route_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    T, E = int(rng.integers(1, 5)), int(rng.integers(1, 7))
    if seed % 2:
        s = rng.integers(-2, 3, size=(T, E)).astype(np.float32)  # heavy ties
        s[rng.random((T, E)) < 0.3] = -0.0
    else:
        s = rng.standard_normal((T, E)).astype(np.float32)
    for k in range(1, E + 1):
        ids, w = M.route(s, k)
        for t in range(T):
            order = _brute_order([float(v) for v in s[t]])
            assert ids[t].tolist() == order[:k]
            sel, rest = set(order[:k]), set(order[k:])
            for i in sel:
                for j in rest:
                    assert s[t, i] > s[t, j] or (s[t, i] == s[t, j] and i < j)
        assert np.all(np.abs(w.sum(axis=1) - 1.0) < 1e-6)
        assert np.all(np.diff(w, axis=1) <= 0)


def test_route_goldens():
    cases = json.load(open(os.path.join(GOLD, "route_small.json")))["cases"]
    for c in cases:
        ids, w = M.route(np.array(c["scores"], dtype=np.float32), c["k"])
        assert ids.tolist() == c["ids"]
        if c["w"] is not None:
            assert w.tolist() == c["w"]


def test_route_k1_is_argmax_with_unit_weight():
    rng = np.random.default_rng(3)
    s = rng.integers(-3, 4, size=(200, 17)).astype(np.float32)
    ids, w = M.route(s, 1)
    assert np.array_equal(ids[:, 0], np.argmax(s, axis=1))  # numpy argmax: first max
    assert np.all(w == 1.0)


def test_route_k_equals_E_is_full_descending_order():
    rng = np.random.default_rng(4)
    s = rng.standard_normal((50, 9)).astype(np.float32)
    ids, _ = M.route(s, 9)
    for t in range(50):
        assert sorted(ids[t].tolist()) == list(range(9))
        assert np.all(np.diff(s[t, ids[t]]) <= 0)


def test_softmax_two_experts_is_logistic():
    rng = np.random.default_rng(5)
    s = rng.standard_normal((300, 6)).astype(np.float32) * 3
    ids, w = M.route(s, 2)
    for t in range(300):
        d = float(s[t, ids[t, 0]]) - float(s[t, ids[t, 1]])
        w0 = 1.0 / (1.0 + math.exp(-d))
        assert abs(w[t, 0] - w0) <= 1e-7
        assert abs(w[t, 1] - (1.0 - w0)) <= 1e-7


def _ids_random(rng, T, E, k, skew=False):
    ids = np.empty((T, k), dtype=np.int32)
    p = None
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p[-3:] = 0
        p /= p.sum()
    for t in range(T):
        ids[t] = rng.choice(E, size=k, replace=False, p=p)
    return ids


@pytest.mark.parametrize("T,E,k,skew", [(1, 8, 2, False), (37, 16, 8, False), (500, 128, 8, True),
                                        (64, 192, 8, False), (257, 8, 8, False)])
def test_shuffle_two_implementations_agree(T, E, k, skew):
    rng = np.random.default_rng(T * 7 + E)
    ids = _ids_random(rng, T, E, k, skew)
    a = M.shuffle(ids, E)
    b = M.shuffle_by_counting(ids, E)
    for x, y in zip(a, b):
        assert x.dtype == np.int32 and np.array_equal(x, y)


@pytest.mark.parametrize("T,E,k", [(300, 32, 4), (1000, 128, 8)])
def test_shuffle_invariants(T, E, k):
    rng = np.random.default_rng(11)
    ids = _ids_random(rng, T, E, k, skew=True)
    counts, offsets, perm, inv = M.shuffle(ids, E)
    R = T * k
    flat = ids.reshape(-1)
    assert counts.sum() == R and offsets[-1] == R and offsets[0] == 0
    assert np.array_equal(np.sort(perm), np.arange(R))
    assert np.array_equal(inv[perm], np.arange(R))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)  # stable: route (token) order kept


def test_shuffle_and_tiles_golden():
    g = json.load(open(os.path.join(GOLD, "shuffle_tiles_small.json")))
    counts, offsets, perm, inv = M.shuffle(np.array(g["ids"], dtype=np.int32), g["E"])
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert perm.tolist() == g["perm"]
    assert inv.tolist() == g["inv"]
    assert M.tile_map(counts, g["BM"]).tolist() == g["tiles"]


@pytest.mark.parametrize("BM", [1, 3, 128])
def test_tile_map_covers_each_row_once(BM):
    rng = np.random.default_rng(BM)
    counts = rng.integers(0, 400, size=40).astype(np.int32)
    counts[[3, 17, 39]] = 0
    offsets = np.concatenate([[0], np.cumsum(counts)])
    tiles = M.tile_map(counts, BM)
    assert len(tiles) == sum(-(-int(c) // BM) for c in counts)
    seen = np.zeros(offsets[-1], dtype=np.int32)
    for e, r0, n in tiles.tolist():
        assert counts[e] > 0 and 1 <= n <= BM
        assert offsets[e] <= r0 and r0 + n <= offsets[e + 1]
        seen[r0:r0 + n] += 1
    assert np.all(seen == 1)
    assert set(tiles[:, 0].tolist()) == {e for e in range(40) if counts[e] > 0}
