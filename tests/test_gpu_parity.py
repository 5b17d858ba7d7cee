"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Integer results (routing ids, counts, offsets, perm, inv, tiles) must match
bit for bit; router weights within 1e-6 (fp32 expf vs fp64 exp); y within
relative L2 <= 1e-2 (bf16) or <= 2e-2 with cosine >= 0.999 (FP8), the
tolerances the method's accuracy targets state ("perf: add small-batch route
MMA for MoE", Correctness: worst relative L2 1.47-1.61%, minimum cosine
0.99987 against a reference)."""
import functools

import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe as O
from oracle.formats import f32_from_bf16_bits
from tests._util import bits16, cosine, oracle_args, rel_l2

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    import __graft_entry__

    __graft_entry__.build()
    import mixture_experts_layer_index_gb300 as mod

    return mod


def _dev(inp):
    return {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}


def _view(ws, addr, n, dtype):
    off = addr - ws.data_ptr()
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


def run_forward(m, wl, d, path=None, ws=None, stream=None):
    path = m.MOE_PATH_AUTO if path is None else path
    p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant, path)
    if ws is None:
        ws = torch.empty(m.moe_workspace_size(p), dtype=torch.uint8, device=DEV)
    y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    m.moe_forward(p, d["x"], d["scores"], d["w1"], d["w2"], d["w1_scale"], d["w2_scale"], y, ws, stream=stream)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(ws) == m.MOE_OK
    return p, y, ws


# ----------------------------------------------------------------------------- routing
def _route_case(m, scores, k):
    T, E = scores.shape
    s = torch.from_numpy(scores).to(DEV)
    ids = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, k, dtype=torch.float32, device=DEV)
    m.moe_route(s, T, E, k, ids, w)
    torch.cuda.synchronize()
    rid, rw = O.route(scores, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    wg = w.cpu().numpy()
    assert np.max(np.abs(wg - rw)) <= 1e-6
    if k == 1:
        assert np.all(wg == 1.0)


@pytest.mark.parametrize("T,E,k", [(16, 8, 2), (4096, 16, 8), (8, 192, 8), (333, 128, 8), (5, 512, 32),
                                   (7, 32, 32), (100, 33, 1), (1, 1, 1), (3, 97, 5)])
def test_route_bit_exact_random(m, T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    _route_case(m, rng.standard_normal((T, E)).astype(np.float32), k)


@pytest.mark.parametrize("E,k", [(8, 2), (64, 8), (300, 17)])
def test_route_ties_and_signed_zeros(m, E, k):
    rng = np.random.default_rng(E)
    s = rng.integers(-2, 3, size=(257, E)).astype(np.float32)
    s[rng.random(s.shape) < 0.3] = -0.0
    s[rng.random(s.shape) < 0.1] = 0.0
    _route_case(m, s, k)


def test_route_full_prefill_skew(m):
    wl = W.workload("prefill")
    _route_case(m, W.make_scores(wl).numpy(), wl.k)


# ----------------------------------------------------------------------------- shuffle
def _ids_random(rng, T, E, k, skew):
    p = None
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p[-4:] = 0
        p /= p.sum()
    keys = rng.random((T, E)) if p is None else rng.random((T, E)) ** (1.0 / np.maximum(p, 1e-30))
    return np.argsort(-keys, axis=1)[:, :k].astype(np.int32)


@pytest.mark.parametrize("T,E,k,skew", [(16, 8, 2, False), (1, 8, 8, False), (129, 16, 8, True),
                                        (16384, 128, 8, True), (2500, 512, 3, False), (1000, 5, 5, False),
                                        (4096, 16, 8, False)])
def test_shuffle_bit_exact(m, T, E, k, skew):
    rng = np.random.default_rng(T + E + k)
    ids = _ids_random(rng, T, E, k, skew)
    R = T * k
    d_ids = torch.from_numpy(ids).to(DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(R, dtype=torch.int32, device=DEV)
    inv = torch.empty(R, dtype=torch.int32, device=DEV)
    ws = torch.empty(m.moe_shuffle_workspace_size(T, E, k), dtype=torch.uint8, device=DEV)
    m.moe_shuffle(d_ids, T, E, k, counts, offsets, perm, inv, ws)
    assert m.moe_read_device_status(ws) == m.MOE_OK
    rc, ro, rp, ri = O.shuffle(ids, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(inv.cpu().numpy(), ri)


def test_shuffle_out_of_range_id_is_reported(m):
    T, E, k = 40, 8, 2
    ids = _ids_random(np.random.default_rng(1), T, E, k, False)
    ids[7, 1] = E  # invalid
    R = T * k
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.full((R,), -7, dtype=torch.int32, device=DEV)
    inv = torch.empty(R, dtype=torch.int32, device=DEV)
    ws = torch.empty(m.moe_shuffle_workspace_size(T, E, k), dtype=torch.uint8, device=DEV)
    m.moe_shuffle(torch.from_numpy(ids).to(DEV), T, E, k, counts, offsets, perm, inv, ws)
    assert m.moe_read_device_status(ws) == m.MOE_ERR_DEVICE_BOUNDS
    assert int(counts.sum()) == R - 1 and inv[15].item() == -1


@pytest.mark.parametrize("BM", [128, 3, 1])
def test_tile_map_bit_exact(m, BM):
    rng = np.random.default_rng(BM)
    counts = rng.integers(0, 700, size=128).astype(np.int32)
    counts[[0, 5, 127]] = 0
    ref = O.tile_map(counts, BM)
    max_tiles = int(counts.sum()) // BM + 128
    tiles = torch.full((max_tiles, 4), -1, dtype=torch.int32, device=DEV)
    nt = torch.empty(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(m.moe_shuffle_workspace_size(0, 128, 1), dtype=torch.uint8, device=DEV)
    m.moe_tile_map(torch.from_numpy(counts).to(DEV), 128, BM, tiles, nt, max_tiles, ws)
    assert m.moe_read_device_status(ws) == m.MOE_OK
    n = nt.item()
    assert n == len(ref)
    assert np.array_equal(tiles[:n, :3].cpu().numpy(), ref)


def test_tile_map_overflow_reports_needed_count(m):
    counts = np.full(16, 300, dtype=np.int32)
    tiles = torch.zeros((5, 4), dtype=torch.int32, device=DEV)
    nt = torch.empty(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(m.moe_shuffle_workspace_size(0, 16, 1), dtype=torch.uint8, device=DEV)
    m.moe_tile_map(torch.from_numpy(counts).to(DEV), 16, 128, tiles, nt, 5, ws)
    assert m.moe_read_device_status(ws) == m.MOE_ERR_DEVICE_BOUNDS
    assert nt.item() == 16 * 3


# ----------------------------------------------------------------------------- forward
def _check_y(wl, y, ref_y, tokens=None):
    got = y.float().cpu().numpy()
    if tokens is not None:
        got = got[tokens]
    assert np.all(np.isfinite(got))
    err = rel_l2(got, ref_y)
    if wl.quant == W.QUANT_BF16:
        assert err <= 1e-2, err
    else:
        assert err <= 2e-2, err
        assert cosine(got, ref_y) >= 0.999
    return err


def _check_quant_views(m, wl, p, ws, inp, ref, opt=None):
    """The activations the Gate/Up GEMM reads, bit for bit: x rows (bf16 copies or
    e4m3 codes) in expert-sorted order on the grouped path, in token order on the
    route-direct path, with their per-(row, 128) scales (blockwise) or the amax of
    x (per tensor).  The quantisation of x is unique (IEEE division by the fp32
    scale, round to nearest even, saturating), so nothing here has a tolerance."""
    v = m.moe_forward_views_ex(p, opt, ws)
    T, H, R = wl.T, wl.H, wl.T * wl.k
    S = opt.n_shared if opt is not None else 0
    xb = bits16(inp["x"])
    grouped = v.perm is not None
    # grouped: the routes' rows in sorted order, then each shared expert's T rows in token order
    rows = np.concatenate([ref["perm"] // wl.k, np.tile(np.arange(T), S)]) if grouped else np.arange(T)
    n = R + S * T if grouped else T
    if wl.quant == W.QUANT_BF16:
        if not v.xs:  # the variant that gathers x inside the GEMM keeps no sorted copy
            return
        got = _view(ws, v.xs, n * H, torch.int16).cpu().numpy().view(np.uint16).reshape(n, H)
        assert np.array_equal(got, xb[rows])
        return
    xf = f32_from_bf16_bits(xb)
    got = _view(ws, v.xs, n * H, torch.uint8).cpu().numpy().reshape(n, H)
    if wl.quant == W.QUANT_FP8_TENSOR:
        amax = np.float32(np.abs(xf).max())
        got_amax = _view(ws, v.amax_x, 1, torch.float32).cpu().numpy()[0]
        assert got_amax.view(np.uint32) == amax.view(np.uint32), (got_amax, amax)
        codes, _ = O.quant_per_tensor(xf)
        assert not v.x_scale
    elif wl.quant == W.QUANT_MXFP8:
        from oracle import mx as OX

        codes, scales = OX.mx_quantize(xf)
        got_s = _view(ws, v.x_scale, n * (H // 32), torch.uint8).cpu().numpy().reshape(n, H // 32)
        assert np.array_equal(got_s, scales[rows])
        assert not v.amax_x
    else:
        codes, scales = O.quant_per_group(xf)
        got_s = _view(ws, v.x_scale, n * (H // 128), torch.float32).cpu().numpy().reshape(n, H // 128)
        assert np.array_equal(got_s.view(np.uint32), scales[rows].view(np.uint32))
        assert not v.amax_x
    bad = got != codes[rows]
    assert not bad.any(), f"{int(bad.sum())} e4m3 codes differ, first at {np.argwhere(bad)[0]}"


def _check_routing_views(m, wl, p, ws, ref, inp=None, opt=None):
    if inp is not None:
        _check_quant_views(m, wl, p, ws, inp, ref, opt)
    v = m.moe_forward_views_ex(p, opt, ws)
    R = wl.T * wl.k
    assert np.array_equal(_view(ws, v.ids, R, torch.int32).cpu().numpy().reshape(wl.T, wl.k), ref["ids"])
    assert np.max(np.abs(_view(ws, v.w, R, torch.float32).cpu().numpy().reshape(wl.T, wl.k) - ref["w"])) <= 1e-6
    if v.perm:
        assert np.array_equal(_view(ws, v.counts, wl.E, torch.int32).cpu().numpy(), ref["counts"])
        assert np.array_equal(_view(ws, v.offsets, wl.E + 1, torch.int32).cpu().numpy(), ref["offsets"])
        assert np.array_equal(_view(ws, v.perm, R, torch.int32).cpu().numpy(), ref["perm"])
        assert np.array_equal(_view(ws, v.inv, R, torch.int32).cpu().numpy(), ref["inv"])
        nt = _view(ws, v.num_tiles, 1, torch.int32).item()
        tiles = _view(ws, v.tiles, nt * 4, torch.int32).cpu().numpy().reshape(nt, 4)[:, :3]
        S = opt.n_shared if opt is not None else 0
        # the shared experts' tiles follow the routed ones: expert E + s, rows T*k + s*T + [0, T)
        shared_tiles = O.tile_map(np.full(S, wl.T, np.int32), m.GEMM_BM) + np.array([wl.E, R, 0], np.int32)
        assert np.array_equal(tiles, np.concatenate([O.tile_map(ref["counts"], m.GEMM_BM), shared_tiles]))


SMALL_GROUPED = [
    W.workload("tiny"),
    W.Workload("ragged", 37, 5, 3, 192, 192, W.QUANT_BF16, 21),   # partial N tiles, 3 K blocks
    W.Workload("dense1", 50, 1, 1, 256, 128, W.QUANT_BF16, 22),   # E = 1, k = 1: dense SwiGLU
    W.Workload("onetok", 1, 16, 8, 512, 256, W.QUANT_BF16, 23),
    W.Workload("kEqE", 20, 4, 4, 128, 64, W.QUANT_BF16, 24),
    W.Workload("tails", 300, 6, 2, 320, 320, W.QUANT_BF16, 25),   # counts not multiples of 128
    # k = 32 (the largest top-k) and an x row of 544 16-byte pieces: more than one pass
    # of the per-token scatter's 256 threads, and eight 4-row batches in the combine
    W.Workload("bigk", 40, 64, 32, 4352, 256, W.QUANT_BF16, 26),
]


@pytest.mark.parametrize("wl", SMALL_GROUPED, ids=lambda w: w.name)
def test_forward_grouped_small_full(m, wl):
    inp = W.make_inputs(wl)
    p, y, ws = run_forward(m, wl, _dev(inp))
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


def test_forward_one_expert_takes_everything(m):
    wl = W.Workload("hot", 700, 8, 2, 256, 128, W.QUANT_BF16, 26)
    inp = W.make_inputs(wl)
    inp["scores"][:, 3] += 100.0  # every token picks expert 3 first: 6 tiles of one expert
    p, y, ws = run_forward(m, wl, _dev(inp))
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    assert ref["counts"][3] == wl.T
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


@functools.lru_cache(maxsize=2)
def _big_inputs(name):
    wl = W.workload(name)
    return wl, W.make_inputs(wl)


@pytest.mark.parametrize("name", ["world16", "prefill"])
def test_forward_grouped_full_size_sampled(m, name):
    wl, inp = _big_inputs(name)
    p, y, ws = run_forward(m, wl, _dev(inp))
    rng = np.random.default_rng(5)
    tokens = np.sort(rng.choice(wl.T, size=192, replace=False))
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant, tokens=tokens)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"], tokens)


@functools.lru_cache(maxsize=1)
def _big_fp8_inputs(quant):
    import dataclasses

    wl = dataclasses.replace(W.workload("prefill"), quant=quant, name=f"prefill_{quant}")
    return wl, W.make_inputs(wl)


@pytest.mark.parametrize("quant", [W.QUANT_FP8_TENSOR, W.QUANT_FP8_BLOCK])
def test_forward_grouped_fp8_full_size_sampled(m, quant):
    """Both FP8 modes at the size their prefill throughput is quoted at (T=16384,
    E=128, top-8, H=2048, I=768, Zipf-skewed): routing views and every quantised x
    row bit-exact, y on 192 sampled tokens.  The oracle's per-tensor h scale is
    taken over all routes (it computes every route's activation for that)."""
    wl, inp = _big_fp8_inputs(quant)
    _big_inputs.cache_clear()
    p, y, ws = run_forward(m, wl, _dev(inp), path=m.MOE_PATH_GROUPED)
    rng = np.random.default_rng(6)
    tokens = np.sort(rng.choice(wl.T, size=192, replace=False))
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant, tokens=tokens)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"], tokens)


def _crafted_x(T, H, quant, seed):
    """x whose quantisation exercises every rounding case of the e4m3 conversion:
    each scale is a power of two (the amax of each scale group is 448 * 2^m), so
    x / s lands exactly on every e4m3 code, on every midpoint between neighbouring
    codes (ties to even), one bf16 step either side of each midpoint, in the
    subnormal range, on +-0.0 and on the amax itself (448)."""
    from oracle.formats import E4M3_VALUES

    mags = np.unique(np.abs(E4M3_VALUES[:0x7F].astype(np.float64)))  # 0 .. 448, 127 magnitudes
    mids = (mags[:-1] + mags[1:]) / 2.0
    step = lambda v: np.ldexp(1.0, np.frexp(v)[1] - 8)  # one bf16 ulp at v (v > 0)
    vals = np.concatenate([mags, mids, mids + step(mids), mids - step(mids)])
    vals = np.concatenate([vals, -vals, [0.0, -0.0]])
    rng = np.random.default_rng(seed)
    x = np.empty((T, H), dtype=np.float64)
    group = {W.QUANT_FP8_TENSOR: H, W.QUANT_MXFP8: 32}.get(quant, 128)
    for t in range(T):
        order = rng.permutation(vals.size)
        pos = 0
        for g0 in range(0, H, group):
            mexp = 0 if quant == W.QUANT_FP8_TENSOR else int(rng.integers(-3, 4))
            seg = np.empty(group)
            seg[0] = 448.0
            take = order[pos:pos + group - 1]
            pos += group - 1
            if take.size < group - 1:  # wrap around when the row is longer than the value list
                extra = rng.permutation(vals.size)[:group - 1 - take.size]
                take = np.concatenate([take, extra])
            seg[1:] = vals[take]
            x[t, g0:g0 + group] = np.ldexp(seg, mexp)
    xt = torch.from_numpy(x).float().to(torch.bfloat16)
    assert torch.equal(xt.double(), torch.from_numpy(x))  # every crafted value is exact in bf16
    return xt


@pytest.mark.parametrize("quant,path", [(W.QUANT_FP8_TENSOR, "grouped"), (W.QUANT_FP8_TENSOR, "route_direct"),
                                        (W.QUANT_FP8_BLOCK, "grouped"), (W.QUANT_FP8_BLOCK, "route_direct"),
                                        (W.QUANT_MXFP8, "grouped")])
def test_fp8_conversion_sweep_through_forward(m, quant, path):
    """The e4m3 conversion of x (cvt.rn.satfinite) against the oracle's encoder on
    every code, midpoint, near-midpoint, subnormal and signed zero, driven through
    moe_forward on both paths: codes and scales bit-exact, y within tolerance."""
    wl = W.Workload(f"cvt_{quant}_{path}", 6, 8, 2, 1024, 128, quant, 70)
    inp = W.make_inputs(wl)
    inp["x"] = _crafted_x(wl.T, wl.H, quant, seed=71)
    xv = inp["x"].double().numpy()
    # every scale group's amax is 448 * 2^m, so every scale amax / 448 is a power of two
    amax = np.abs(xv).reshape(wl.T, -1, {W.QUANT_FP8_TENSOR: wl.H, W.QUANT_MXFP8: 32}.get(quant, 128)).max(axis=2)
    assert np.all(np.frexp(amax / 448.0)[0] == 0.5)
    mp = m.MOE_PATH_GROUPED if path == "grouped" else m.MOE_PATH_ROUTE_DIRECT
    p, y, ws = run_forward(m, wl, _dev(inp), path=mp)
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


@functools.lru_cache(maxsize=1)
def _decode_weights(name):
    wl = W.workload(name, 1)
    return W.make_weights(wl)


@pytest.mark.parametrize("B", range(1, 9))
@pytest.mark.parametrize("name", W.DECODE_SWEEPS)
def test_forward_route_direct_decode(m, name, B):
    wl = W.workload(name, B)
    w1, w2, s1, s2 = _decode_weights(name)
    inp = {"x": W.make_x(wl), "scores": W.make_scores(wl), "w1": w1, "w2": w2, "w1_scale": s1, "w2_scale": s2}
    p, y, ws = run_forward(m, wl, _dev(inp))
    assert m.moe_select_path(p) == m.MOE_PATH_ROUTE_DIRECT
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


@pytest.mark.parametrize("quant", [W.QUANT_FP8_TENSOR, W.QUANT_FP8_BLOCK])
@pytest.mark.parametrize("T", [1, 9, 64, 128])
def test_forward_route_direct_shapes(m, quant, T):
    # more tokens than one MMA's 8 columns share an expert; up to the 1024-route limit
    wl = W.Workload(f"rd{T}", T, 24, 8, 256, 256, quant, 30 + T)
    inp = W.make_inputs(wl)
    p, y, ws = run_forward(m, wl, _dev(inp), path=m.MOE_PATH_ROUTE_DIRECT)
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


@pytest.mark.parametrize("wl", [W.workload("tiny"), W.workload("hunyuan", 4), W.workload("qwen3a", 3),
                                W.Workload("f8t_det", 200, 32, 8, 512, 256, W.QUANT_FP8_TENSOR, 61),
                                W.Workload("f8b_det", 200, 32, 8, 512, 256, W.QUANT_FP8_BLOCK, 62)],
                         ids=lambda w: w.name)
def test_deterministic_and_graph_replay_bitwise(m, wl):
    if wl.name.split("_")[0] not in W.DECODE_SWEEPS:
        inp = W.make_inputs(wl)
    else:
        w1, w2, s1, s2 = _decode_weights(wl.name.split("_")[0])
        inp = {"x": W.make_x(wl), "scores": W.make_scores(wl), "w1": w1, "w2": w2, "w1_scale": s1, "w2_scale": s2}
    d = _dev(inp)
    p, y1, ws = run_forward(m, wl, d)
    _, y2, _ = run_forward(m, wl, d, ws=ws)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    # capture one forward in a CUDA graph (preallocated output and workspace) and replay it
    y3 = torch.empty_like(y1)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        m.moe_forward(p, d["x"], d["scores"], d["w1"], d["w2"], d["w1_scale"], d["w2_scale"], y3, ws,
                      stream=s)
    for _ in range(3):
        y3.fill_(0)
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))


def test_empty_batch_leaves_output_untouched(m):
    p = m.problem(0, 8, 2, 256, 128)
    m.moe_forward(p, None, None, None, None, None, None, None, None, 0)


def test_profile_single_stage_and_all_stages(m):
    # moe_profile_start_stage times only the named stage; moe_profile_start times all
    wl = W.Workload("prof", 300, 16, 4, 256, 128, W.QUANT_BF16, 27)
    d = _dev(W.make_inputs(wl))
    m.moe_profile_start_stage("gateup_gemm")
    for _ in range(3):
        run_forward(m, wl, d)
    st = m.moe_profile_stop()
    assert set(st) == {"gateup_gemm"} and st["gateup_gemm"][1] == 3 and st["gateup_gemm"][0] > 0
    m.moe_profile_start()
    run_forward(m, wl, d)
    st = m.moe_profile_stop()
    assert {"route_rank", "scan_tiles", "scatter_gather", "gateup_gemm", "down_gemm", "combine"} <= set(st)
    assert all(n == 1 for _, n in st.values())


def test_small_workspace_rejected_without_launch(m):
    wl = W.workload("tiny")
    d = _dev(W.make_inputs(wl))
    p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I)
    need = m.moe_workspace_size(p)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    y = torch.full((wl.T, wl.H), 7.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(m.MoeError) as ei:
        m.moe_forward(p, d["x"], d["scores"], d["w1"], d["w2"], None, None, y, ws, ws_bytes=need - 1)
    assert ei.value.status == m.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


FP8_GROUPED = [
    W.Workload("f8g_small", 64, 32, 8, 512, 256, W.QUANT_FP8_TENSOR, 41),
    W.Workload("f8g_ragged", 300, 16, 4, 384, 192, W.QUANT_FP8_TENSOR, 42),  # partial N tile, Down K tail
    W.Workload("f8g_tiny", 5, 8, 2, 256, 128, W.QUANT_FP8_TENSOR, 43),
]


@pytest.mark.parametrize("wl", FP8_GROUPED, ids=lambda w: w.name)
def test_forward_grouped_fp8_per_tensor(m, wl):
    inp = W.make_inputs(wl)
    p, y, ws = run_forward(m, wl, _dev(inp), path=m.MOE_PATH_GROUPED)
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


def test_forward_grouped_fp8_hunyuan_shape_and_auto_switch(m):
    wl = W.workload("hunyuan", 1).with_tokens(512)
    w1, w2, s1, s2 = _decode_weights("hunyuan")
    inp = {"x": W.make_x(wl), "scores": W.make_scores(wl), "w1": w1, "w2": w2, "w1_scale": s1, "w2_scale": s2}
    p, y, ws = run_forward(m, wl, _dev(inp))
    assert m.moe_select_path(p) == m.MOE_PATH_GROUPED
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])
    assert m.moe_select_path(m.problem(96, wl.E, wl.k, wl.H, wl.I, wl.quant)) == m.MOE_PATH_ROUTE_DIRECT
    assert m.moe_select_path(m.problem(97, wl.E, wl.k, wl.H, wl.I, wl.quant)) == m.MOE_PATH_GROUPED


@pytest.mark.parametrize("name,T", [("hunyuan", 96), ("qwen3a", 64), ("qwen3b", 64)])
def test_forward_auto_route_direct_at_its_largest_batch(m, name, T):
    """The largest batch AUTO sends down the route-direct path, at the decode shapes
    the crossover was measured on: 768 / 512 routes over most of the experts."""
    wl = W.workload(name, 1).with_tokens(T)
    w1, w2, s1, s2 = _decode_weights(name)
    inp = {"x": W.make_x(wl), "scores": W.make_scores(wl), "w1": w1, "w2": w2, "w1_scale": s1, "w2_scale": s2}
    p, y, ws = run_forward(m, wl, _dev(inp))
    assert m.moe_select_path(p) == m.MOE_PATH_ROUTE_DIRECT
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


@pytest.mark.parametrize("T", [4, 24])
def test_fp8_grouped_and_route_direct_agree(m, T):
    wl = W.Workload("f8agree", T, 48, 8, 512, 256, W.QUANT_FP8_TENSOR, 44 + T)
    inp = W.make_inputs(wl)
    d = _dev(inp)
    _, yg, _ = run_forward(m, wl, d, path=m.MOE_PATH_GROUPED)
    _, yr, _ = run_forward(m, wl, d, path=m.MOE_PATH_ROUTE_DIRECT)
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_y(wl, yg, ref["y"])
    _check_y(wl, yr, ref["y"])
    assert rel_l2(yg.float().cpu().numpy(), yr.float().cpu().numpy()) <= 2e-2


FP8_BLOCK_GROUPED = [
    W.Workload("f8b_small", 64, 32, 8, 512, 256, W.QUANT_FP8_BLOCK, 51),
    # 3 Gate/Up groups of 128 h columns; 2 Down N tiles of 256 columns, the second with 128
    W.Workload("f8b_ragged", 300, 16, 4, 384, 384, W.QUANT_FP8_BLOCK, 52),
    W.Workload("f8b_tiny", 5, 8, 2, 256, 128, W.QUANT_FP8_BLOCK, 53),
    W.Workload("f8b_onexp", 130, 1, 1, 128, 128, W.QUANT_FP8_BLOCK, 54),  # one K block each way, 2 row tiles
    # a last scale group of I with 64 columns (the route-MMA page's dispatch admits I % 64 == 0):
    # half of that Gate/Up group's columns idle, a half K block in the Down GEMM
    W.Workload("f8b_i320", 300, 16, 4, 384, 320, W.QUANT_FP8_BLOCK, 56),
    W.Workload("f8b_i64", 70, 8, 2, 256, 64, W.QUANT_FP8_BLOCK, 58),
]


@pytest.mark.parametrize("wl", FP8_BLOCK_GROUPED, ids=lambda w: w.name)
def test_forward_grouped_fp8_blockwise(m, wl):
    inp = W.make_inputs(wl)
    p, y, ws = run_forward(m, wl, _dev(inp), path=m.MOE_PATH_GROUPED)
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


def test_forward_grouped_fp8_blockwise_qwen3_shape_and_auto_switch(m):
    wl = W.workload("qwen3a", 1).with_tokens(512)
    w1, w2, s1, s2 = _decode_weights("qwen3a")
    inp = {"x": W.make_x(wl), "scores": W.make_scores(wl), "w1": w1, "w2": w2, "w1_scale": s1, "w2_scale": s2}
    p, y, ws = run_forward(m, wl, _dev(inp))
    assert m.moe_select_path(p) == m.MOE_PATH_GROUPED
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])
    assert m.moe_select_path(m.problem(64, wl.E, wl.k, wl.H, wl.I, wl.quant)) == m.MOE_PATH_ROUTE_DIRECT
    assert m.moe_select_path(m.problem(65, wl.E, wl.k, wl.H, wl.I, wl.quant)) == m.MOE_PATH_GROUPED


@pytest.mark.parametrize("T", [4, 24])
def test_fp8_blockwise_grouped_and_route_direct_agree(m, T):
    wl = W.Workload("f8bagree", T, 48, 8, 512, 256, W.QUANT_FP8_BLOCK, 55 + T)
    inp = W.make_inputs(wl)
    d = _dev(inp)
    _, yg, _ = run_forward(m, wl, d, path=m.MOE_PATH_GROUPED)
    _, yr, _ = run_forward(m, wl, d, path=m.MOE_PATH_ROUTE_DIRECT)
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_y(wl, yg, ref["y"])
    _check_y(wl, yr, ref["y"])
    assert rel_l2(yg.float().cpu().numpy(), yr.float().cpu().numpy()) <= 2e-2


def test_gather4_variant_matches_oracle_in_subprocess():
    """The fused TMA tile::gather4 Gate/Up variant (selected by MOE_GATEUP_A=gather4,
    read once per process) stays correct; run it in a fresh process."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import __graft_entry__ as g, workloads as W, mixture_experts_layer_index_gb300 as m;"
            "print(g._run_case(W.Workload('g4', 300, 6, 2, 320, 320, W.QUANT_BF16, 25), m.MOE_PATH_GROUPED));"
            "print(g._run_case(W.workload('tiny'), m.MOE_PATH_GROUPED))")
    env = dict(os.environ, MOE_GATEUP_A="gather4")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr


# ----------------------------------------------------------------------------- shared experts, fp32 partials
def _shared_weights(wl, S, seed):
    """S shared experts with the routed experts' shapes and format (own seed)."""
    sw = W.Workload(f"{wl.name}_shared", wl.T, S, 1, wl.H, wl.I, wl.quant, seed)
    w1, w2, s1, s2 = W.make_weights(sw)
    return {"w1": w1, "w2": w2, "w1_scale": s1, "w2_scale": s2}


def _oracle_shared(sh):
    from tests._util import u8

    cv = (lambda t: bits16(t)) if sh["w1"].dtype == torch.bfloat16 else (lambda t: u8(t))
    return {"w1": cv(sh["w1"]), "w2": cv(sh["w2"]),
            "w1_scale": None if sh["w1_scale"] is None else sh["w1_scale"].numpy(),
            "w2_scale": None if sh["w2_scale"] is None else sh["w2_scale"].numpy()}


def run_forward_ex(m, wl, d, shd, S, y_fp32=False, path=None):
    path = m.MOE_PATH_AUTO if path is None else path
    p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant, path)
    opt = m.forward_options(S, shd["w1"], shd["w2"], shd["w1_scale"], shd["w2_scale"], y_fp32)
    ws = torch.empty(m.moe_workspace_size_ex(p, opt), dtype=torch.uint8, device=DEV)
    y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.float32 if y_fp32 else torch.bfloat16, device=DEV)
    m.moe_forward_ex(p, opt, d["x"], d["scores"], d["w1"], d["w2"], d["w1_scale"], d["w2_scale"], y, ws)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(ws) == m.MOE_OK
    return p, opt, y, ws


SHARED_CASES = [
    (W.workload("tiny"), 1, None),
    (W.Workload("sh_ragged", 300, 6, 2, 320, 320, W.QUANT_BF16, 81), 2, None),   # partial tiles, 2 shared
    (W.workload("world16"), 1, 192),
    (W.workload("prefill"), 1, 192),
    (W.Workload("sh_f8t", 200, 16, 4, 512, 256, W.QUANT_FP8_TENSOR, 82), 1, None),
    (W.Workload("sh_f8b", 200, 16, 4, 512, 256, W.QUANT_FP8_BLOCK, 83), 2, None),
]


@pytest.mark.parametrize("wl,S,sample", SHARED_CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_forward_shared_experts(m, wl, S, sample):
    """Shared experts ("shared output", route-MMA page, Summary) through
    moe_forward_ex: every token's row of every shared expert joins the grouped
    GEMMs as expert E + s; y = routed sum + shared outputs, rounded once."""
    inp = _big_inputs(wl.name)[1] if wl.name in ("world16", "prefill") else W.make_inputs(wl)
    shd = _shared_weights(wl, S, 500 + S)
    d = _dev(inp)
    p, opt, y, ws = run_forward_ex(m, wl, d, _dev(shd), S)
    tokens = None
    if sample:
        tokens = np.sort(np.random.default_rng(8).choice(wl.T, size=sample, replace=False))
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant, tokens=tokens, shared=_oracle_shared(shd))
    _check_routing_views(m, wl, p, ws, ref, inp, opt)
    _check_y(wl, y, ref["y"], tokens)
    # the shared term matters: without it the result is far from the reference
    ref0 = O.forward(*oracle_args(inp), wl.k, wl.quant, tokens=tokens)
    assert rel_l2(ref0["y"], ref["y"]) > 0.1


def test_route_direct_with_shared_experts_is_rejected(m):
    wl = W.workload("hunyuan", 2)
    p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant, m.MOE_PATH_ROUTE_DIRECT)
    opt = m.forward_options(1, 16, 16, 4, 4)  # never dereferenced: rejected before any launch
    assert m.moe_workspace_size_ex(p, opt) == 0
    assert m.moe_workspace_size_ex(m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant), opt) > 0


@pytest.mark.parametrize("quant,path", [(W.QUANT_BF16, "grouped"), (W.QUANT_FP8_TENSOR, "grouped"),
                                        (W.QUANT_FP8_BLOCK, "grouped"), (W.QUANT_FP8_TENSOR, "route_direct"),
                                        (W.QUANT_FP8_BLOCK, "route_direct")])
def test_fp32_partial_output_and_rounding(m, quant, path):
    """y_fp32 = 1 writes the unrounded sum (checked against the oracle's unrounded
    y); moe_round_bf16 of it equals the forward's own bf16 output bit for bit."""
    wl = W.Workload(f"y32_{quant}", 24, 16, 4, 512, 256, quant, 84)
    inp = W.make_inputs(wl)
    d = _dev(inp)
    mp = m.MOE_PATH_GROUPED if path == "grouped" else m.MOE_PATH_ROUTE_DIRECT
    none = {"w1": None, "w2": None, "w1_scale": None, "w2_scale": None}
    _, _, y32, _ = run_forward_ex(m, wl, d, none, 0, y_fp32=True, path=mp)
    _, y16, _ = run_forward(m, wl, d, path=mp)
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant, y_fp32=True)
    got = y32.cpu().numpy()
    assert rel_l2(got, ref["y"]) <= (1e-2 if quant == W.QUANT_BF16 else 2e-2)
    yr = torch.empty_like(y16)
    m.moe_round_bf16(y32, yr)
    torch.cuda.synchronize()
    assert torch.equal(yr.view(torch.int16), y16.view(torch.int16))
    assert torch.equal(yr.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))  # RNE, as torch rounds


@pytest.mark.parametrize("quant", [W.QUANT_BF16, W.QUANT_FP8_BLOCK])
def test_tensor_parallel_slices_on_gpu(m, quant):
    """Two slices of a tensor-parallel split of I, each run as its own forward
    with y_fp32 = 1 (one per rank in a TP deployment, here one after the other on
    one GPU), summed and rounded once with moe_round_bf16: equal to the unsplit
    forward's oracle within the usual tolerance, shared expert included."""
    from mixture_experts_layer_index_gb300.tp import shard_weights

    wl = W.Workload(f"tp_{quant}", 200, 16, 4, 512, 256, quant, 85)
    inp = W.make_inputs(wl)
    shd = _shared_weights(wl, 1, 86)
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant, shared=_oracle_shared(shd))
    P = 2
    acc = torch.zeros(wl.T, wl.H, dtype=torch.float32, device=DEV)
    sl = W.Workload(wl.name + "_slice", wl.T, wl.E, wl.k, wl.H, wl.I // P, quant, 85)
    for rank in range(P):
        w1, w2, s1, s2 = shard_weights(inp["w1"], inp["w2"], inp["w1_scale"], inp["w2_scale"], quant, rank, P)
        c1, c2, d1, d2 = shard_weights(shd["w1"], shd["w2"], shd["w1_scale"], shd["w2_scale"], quant, rank, P)
        part_in = {"x": inp["x"], "scores": inp["scores"], "w1": w1, "w2": w2, "w1_scale": s1, "w2_scale": s2}
        part_sh = {"w1": c1, "w2": c2, "w1_scale": d1, "w2_scale": d2}
        _, _, y32, _ = run_forward_ex(m, sl, _dev(part_in), _dev(part_sh), 1, y_fp32=True, path=m.MOE_PATH_GROUPED)
        acc += y32
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=DEV)
    m.moe_round_bf16(acc, y)
    torch.cuda.synchronize()
    _check_y(wl, y, ref["y"])


# ----------------------------------------------------------------------------- MXFP8
def _mx_group_case(m, rows, cols, sizes, seed):
    from oracle import mx as OX

    rng = np.random.default_rng(seed)
    sc = rng.integers(0, 255, size=(rows, cols)).astype(np.uint8)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    assert off[-1] <= rows
    G = len(sizes)
    out = torch.full((m.moe_mx_blocked_bytes(rows, cols, G),), 0xAB, dtype=torch.uint8, device=DEV)
    starts = torch.full((G + 1,), -1, dtype=torch.int32, device=DEV)
    ws = torch.empty(m.moe_mx_blocked_workspace_size(rows, G), dtype=torch.uint8, device=DEV)
    m.moe_mx_blocked_scales(torch.from_numpy(sc).to(DEV), rows, cols, torch.from_numpy(off).to(DEV), G, out, starts, ws)
    assert m.moe_read_device_status(ws) == m.MOE_OK
    ref, ref_starts = OX.per_group_blocked(sc, off)
    assert np.array_equal(starts.cpu().numpy(), ref_starts)
    got = out.cpu().numpy()[:ref.size].reshape(ref.shape)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("rows,cols,sizes", [
    (16640, 160, [1040] * 16),                           # the page's benchmark shape, 16 groups
    (700, 5, [3, 0, 130, 128, 400]),                     # ragged, an empty group, cols not a multiple of 4
    (2048, 64, [0, 0, 2048]),
    (131072, 24, list(np.random.default_rng(3).multinomial(131072, np.ones(128) / 128))),
    (1, 1, [1]),
])
def test_mx_blocked_scales_bit_exact(m, rows, cols, sizes):
    """The per-group blocked scale conversion ("[mxfp8 moe training] add per group
    blocked scale kernels") against the oracle, byte for byte, with the groups'
    padded start rows computed on the device."""
    _mx_group_case(m, rows, cols, [int(v) for v in sizes], rows + cols)


def test_mx_blocked_scales_reports_groups_outside_the_matrix(m):
    rows, cols = 300, 8
    off = torch.tensor([0, 100, 400], dtype=torch.int32, device=DEV)  # second group runs past the last row
    out = torch.zeros(m.moe_mx_blocked_bytes(rows, cols, 2), dtype=torch.uint8, device=DEV)
    starts = torch.zeros(3, dtype=torch.int32, device=DEV)
    ws = torch.empty(m.moe_mx_blocked_workspace_size(rows, 2), dtype=torch.uint8, device=DEV)
    m.moe_mx_blocked_scales(torch.zeros(rows, cols, dtype=torch.uint8, device=DEV), rows, cols, off, 2, out, starts, ws)
    assert m.moe_read_device_status(ws) == m.MOE_ERR_DEVICE_BOUNDS
    assert starts.cpu().tolist() == [0, 128, 128]


MX_GROUPED = [
    W.Workload("mx_small", 64, 32, 8, 512, 256, W.QUANT_MXFP8, 101),
    W.Workload("mx_ragged", 300, 16, 4, 384, 192, W.QUANT_MXFP8, 102),   # I % 128 == 64: a half K stage in Down
    W.Workload("mx_tiny", 5, 8, 2, 256, 128, W.QUANT_MXFP8, 103),
    W.Workload("mx_dense", 130, 1, 1, 128, 64, W.QUANT_MXFP8, 104),    # E = k = 1, two row tiles, one K stage
]


@pytest.mark.parametrize("wl", MX_GROUPED, ids=lambda w: w.name)
def test_forward_grouped_mxfp8(m, wl):
    inp = W.make_inputs(wl)
    p, y, ws = run_forward(m, wl, _dev(inp))
    assert m.moe_select_path(p) == m.MOE_PATH_GROUPED
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


def test_forward_mxfp8_with_shared_experts_and_fp32_partial(m):
    wl = W.Workload("mx_shared", 200, 16, 4, 512, 256, W.QUANT_MXFP8, 105)
    inp = W.make_inputs(wl)
    shd = _shared_weights(wl, 2, 106)
    d = _dev(inp)
    p, opt, y, ws = run_forward_ex(m, wl, d, _dev(shd), 2)
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant, shared=_oracle_shared(shd))
    _check_routing_views(m, wl, p, ws, ref, inp, opt)
    _check_y(wl, y, ref["y"])
    _, _, y32, _ = run_forward_ex(m, wl, d, _dev(shd), 2, y_fp32=True)
    assert torch.equal(y32.to(torch.bfloat16).view(torch.int16), y.view(torch.int16))


def test_forward_grouped_mxfp8_full_size_sampled(m):
    import dataclasses

    wl = dataclasses.replace(W.workload("prefill"), quant=W.QUANT_MXFP8, name="prefill_mxfp8")
    inp = W.make_inputs(wl)
    _big_inputs.cache_clear()
    _big_fp8_inputs.cache_clear()
    p, y, ws = run_forward(m, wl, _dev(inp))
    tokens = np.sort(np.random.default_rng(7).choice(wl.T, size=192, replace=False))
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant, tokens=tokens)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"], tokens)


def test_mxfp8_route_direct_is_rejected(m):
    p = m.problem(2, 16, 4, 256, 128, "mxfp8", m.MOE_PATH_ROUTE_DIRECT)
    assert m.moe_workspace_size(p) == 0
    assert m.moe_select_path(m.problem(2, 16, 4, 256, 128, "mxfp8")) == m.MOE_PATH_GROUPED


@pytest.mark.parametrize("path", ["grouped", "route_direct"])
@pytest.mark.parametrize("wl", [W.Workload("f8b_qwen_i192", 512, 128, 8, 2048, 192, W.QUANT_FP8_BLOCK, 57),
                                W.Workload("f8t_hunyuan_h4032", 512, 192, 8, 4032, 192, W.QUANT_FP8_TENSOR, 47)],
                         ids=lambda w: w.name)
def test_forward_page_admitted_shapes(m, wl, path):
    """Shapes the route-MMA page's dispatch admits beyond this library's first
    limits, on both paths: blockwise FP8 with I % 128 == 64 (a 64-column last scale
    group of h) and per-tensor FP8 with H % 128 == 64 (a half K box at the end of
    every weight row); the route-direct path at decode sizes."""
    if path == "route_direct":
        wl = wl.with_tokens(4)
    inp = W.make_inputs(wl)
    mp = m.MOE_PATH_GROUPED if path == "grouped" else m.MOE_PATH_ROUTE_DIRECT
    p, y, ws = run_forward(m, wl, _dev(inp), path=mp)
    assert m.moe_select_path(m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant)) == mp
    ref = O.forward(*oracle_args(inp), wl.k, wl.quant)
    _check_routing_views(m, wl, p, ws, ref, inp)
    _check_y(wl, y, ref["y"])


def test_mxfp8_weight_scales_converted_once(m):
    """moe_mx_weight_scales converts the weights' scales into the forward's blocked
    layouts once; the forward given them (mx_weight_scales_blocked = 1) must give
    the same y, bit for bit, as the forward that converts on every call, with
    shared experts converted the same way."""
    wl = W.Workload("mx_preblocked", 150, 16, 4, 512, 320, W.QUANT_MXFP8, 107)
    inp = W.make_inputs(wl)
    shd = _shared_weights(wl, 1, 108)
    d, sd = _dev(inp), _dev(shd)
    _, _, y_ref, _ = run_forward_ex(m, wl, d, sd, 1)

    def blocked(w1s, w2s, E):
        b1 = torch.empty(m.moe_mx_weight_scales_bytes(E, wl.H, wl.I, 1), dtype=torch.uint8, device=DEV)
        b2 = torch.empty(m.moe_mx_weight_scales_bytes(E, wl.H, wl.I, 2), dtype=torch.uint8, device=DEV)
        m.moe_mx_weight_scales(w1s, w2s, E, wl.H, wl.I, b1, b2)
        return b1, b2

    b1, b2 = blocked(d["w1_scale"], d["w2_scale"], wl.E)
    c1, c2 = blocked(sd["w1_scale"], sd["w2_scale"], 1)
    p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant)
    opt = m.forward_options(1, sd["w1"], sd["w2"], c1, c2, mx_weight_scales_blocked=True)
    ws = torch.empty(m.moe_workspace_size_ex(p, opt), dtype=torch.uint8, device=DEV)
    y = torch.empty_like(y_ref)
    for _ in range(2):
        y.fill_(0)
        m.moe_forward_ex(p, opt, d["x"], d["scores"], d["w1"], d["w2"], b1, b2, y, ws)
        torch.cuda.synchronize()
        assert m.moe_read_device_status(ws) == m.MOE_OK
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
