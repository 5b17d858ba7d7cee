"""Pins for the oracle's forward pass (all three quantisation modes).

1. Closed form: identity-like experts with top_k = 1.  Gate row i of W1[e] has
   a single nonzero at column sigma_e(i), the up row I+i one at the same
   column with a different coefficient, and row c of W2[e] a single nonzero at
   column pi_e(c mod I).  Every dot product then has one term, so the whole
   forward reduces to the SwiGLU formula applied elementwise; the expected
   value is computed here with math.exp and torch's own bf16 / float8
   conversions.  A swapped gate/up, a transposed or mis-indexed operand, a
   wrong scale block or a dropped scale changes the result.
2. Library special case: E = 1, k = 1 is a dense SwiGLU MLP, computed with
   torch CPU matmuls and F.silu.
3. Brute force: y_t = sum over ALL experts of gate_e(t) * FFN_e(x_t), with
   gate_e(t) the softmax weight when e is selected and 0 otherwise (routing
   by a comparator sort, softmax by math.exp), on tiny inputs.
4. FP8 noise: the quantised forward stays within a few percent of the
   unquantised one, the order of the errors reported for the route-MMA path
   ("perf: add small-batch route MMA for MoE", Correctness: worst relative L2
   1.47% per-tensor, 1.61% blockwise).
"""
import functools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

from oracle import moe as M
from tests._util import bits16, rel_l2

E4 = torch.float8_e4m3fn


def _t_bf16_bits(a64):
    """fp64 numpy -> fp32 -> bf16 (torch conversions) -> uint16 bits."""
    t = torch.from_numpy(np.asarray(a64, dtype=np.float64)).float().to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _t_bf16_val(a64):
    return torch.from_numpy(np.asarray(a64, dtype=np.float64)).float().to(torch.bfloat16).float().numpy()


def _t_e4m3(v32):
    """fp32 numpy -> (code value as fp32) via torch's float8 conversion."""
    return torch.from_numpy(np.asarray(v32, dtype=np.float32)).to(E4).float().numpy()


def _silu_u(g, u):
    return np.array([gi / (1.0 + math.exp(-gi)) * ui for gi, ui in zip(g.ravel(), u.ravel())]).reshape(g.shape)


CODE_1 = 0x38
CODE_2 = 0x40


def _identity_case(quant, T=24, E=4, H=512, I=256, seed=0):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    scores = rng.standard_normal((T, E)).astype(np.float32)
    sig = [rng.permutation(H)[:I] for _ in range(E)]
    pi = [rng.permutation(I) for _ in range(E)]
    alpha = [0.5, 2.0, 1.0, 4.0][:E]
    gamma = [1.0, 0.25, 2.0, 0.5][:E]
    beta = [2.0, 1.0, 0.5, 0.25][:E]
    if quant == M.BF16:
        w1 = torch.zeros(E, 2 * I, H)
        w2 = torch.zeros(E, H, I)
        for e in range(E):
            w1[e, np.arange(I), sig[e]] = alpha[e]
            w1[e, I + np.arange(I), sig[e]] = gamma[e]
            w2[e, np.arange(H), pi[e][np.arange(H) % I]] = beta[e]
        w1, w2 = w1.to(torch.bfloat16), w2.to(torch.bfloat16)
        s1 = s2 = None
        w1n, w2n = bits16(w1), bits16(w2)
    else:
        w1n = np.zeros((E, 2 * I, H), dtype=np.uint8)
        w2n = np.zeros((E, H, I), dtype=np.uint8)
        for e in range(E):
            w1n[e, np.arange(I), sig[e]] = CODE_2
            w1n[e, I + np.arange(I), sig[e]] = CODE_1
            w2n[e, np.arange(H), pi[e][np.arange(H) % I]] = CODE_1
        if quant == M.FP8_TENSOR:
            s1 = np.array(alpha, dtype=np.float32)
            s2 = np.array(beta, dtype=np.float32)
        else:
            s1 = (2.0 ** rng.integers(-3, 4, size=(E, 2 * I // 128, H // 128))).astype(np.float32)
            s2 = (2.0 ** rng.integers(-3, 4, size=(E, H // 128, I // 128))).astype(np.float32)
    return dict(x=x, scores=scores, w1=w1n, w2=w2n, s1=s1, s2=s2, sig=sig, pi=pi,
                alpha=alpha, gamma=gamma, beta=beta, T=T, E=E, H=H, I=I)


def _expected_identity(c, quant):
    T, H, I = c["T"], c["H"], c["I"]
    xv = c["x"].float().numpy()
    e_of = np.argmax(c["scores"], axis=1)  # k = 1, continuous scores: no ties
    a = np.zeros((T, I), dtype=np.float32)
    if quant == M.BF16:
        for t in range(T):
            e = e_of[t]
            xs = xv[t, c["sig"][e]].astype(np.float64)
            a[t] = _silu_u(c["alpha"][e] * xs, c["gamma"][e] * xs)
        h = _t_bf16_val(a).astype(np.float64)
    elif quant == M.FP8_TENSOR:
        sx = np.float32(np.abs(xv).max()) / np.float32(448.0)
        qx = _t_e4m3(xv / sx).astype(np.float64)
        for t in range(T):
            e = e_of[t]
            sc = np.float64(sx) * np.float64(c["s1"][e])
            qs = qx[t, c["sig"][e]]
            a[t] = _silu_u(sc * 2.0 * qs, sc * qs)
        sh = np.float32(np.abs(a).max()) / np.float32(448.0)
        h = _t_e4m3(a / sh).astype(np.float64)
    else:
        ng = H // 128
        sx = np.stack([np.abs(xv[:, g * 128:(g + 1) * 128]).max(axis=1) for g in range(ng)], 1)
        sx = sx.astype(np.float32) / np.float32(448.0)
        qx = _t_e4m3(xv / np.repeat(sx, 128, axis=1)).astype(np.float64)
        for t in range(T):
            e = e_of[t]
            s = c["sig"][e]
            G = s // 128
            i = np.arange(I)
            g = sx[t, G] * c["s1"][e][i // 128, G].astype(np.float64) * 2.0 * qx[t, s]
            u = sx[t, G] * c["s1"][e][(I + i) // 128, G].astype(np.float64) * qx[t, s]
            a[t] = _silu_u(g, u)
        ngi = I // 128
        sh = np.stack([np.abs(a[:, g * 128:(g + 1) * 128]).max(axis=1) for g in range(ngi)], 1)
        sh = sh.astype(np.float32) / np.float32(448.0)
        h = _t_e4m3(a / np.repeat(sh, 128, axis=1)).astype(np.float64)
    y = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        e = e_of[t]
        src = c["pi"][e][np.arange(H) % I]
        if quant == M.BF16:
            y[t] = c["beta"][e] * h[t, src]
        elif quant == M.FP8_TENSOR:
            y[t] = (np.float64(sh) * np.float64(c["s2"][e])) * h[t, src]
        else:
            cidx = np.arange(H)
            y[t] = sh[t, src // 128].astype(np.float64) * c["s2"][e][cidx // 128, src // 128] * h[t, src]
    return _t_bf16_val(y)


@pytest.mark.parametrize("quant", [M.BF16, M.FP8_TENSOR, M.FP8_BLOCK])
def test_identity_experts_closed_form(quant):
    c = _identity_case(quant)
    out = M.forward(bits16(c["x"]), c["scores"], c["w1"], c["w2"], c["s1"], c["s2"], 1, quant)
    exp = _expected_identity(c, quant)
    assert np.all(out["w"] == 1.0)
    assert np.array_equal(out["y"], exp)


def test_identity_closed_form_detects_gate_up_swap():
    # the closed form distinguishes gate from up: swapping the two halves of W1
    # gives a different y (a guard that the pin above has teeth)
    c = _identity_case(M.BF16)
    w1s = np.concatenate([c["w1"][:, c["I"]:], c["w1"][:, :c["I"]]], axis=1)
    out = M.forward(bits16(c["x"]), c["scores"], w1s, c["w2"], None, None, 1, M.BF16)
    assert not np.array_equal(out["y"], _expected_identity(c, M.BF16))


def test_dense_swiglu_single_expert_matches_torch():
    rng = np.random.default_rng(7)
    T, H, I = 40, 256, 192
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    w1 = (torch.from_numpy(rng.standard_normal((1, 2 * I, H)).astype(np.float32)) / math.sqrt(H)).to(torch.bfloat16)
    w2 = (torch.from_numpy(rng.standard_normal((1, H, I)).astype(np.float32)) / math.sqrt(I)).to(torch.bfloat16)
    scores = rng.standard_normal((T, 1)).astype(np.float32)
    out = M.forward(bits16(x), scores, bits16(w1), bits16(w2), None, None, 1, M.BF16)
    X = x.double()
    g = X @ w1[0, :I].double().T
    u = X @ w1[0, I:].double().T
    hh = (Fnn.silu(g) * u).float().to(torch.bfloat16).double()
    y = (hh @ w2[0].double().T).float().to(torch.bfloat16).float().numpy()
    ulp = np.abs(y) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(out["y"] - y) <= ulp)
    assert np.mean(out["y"] == y) > 0.999


def _brute_route(s, k):
    def cmp(i, j):
        if s[i] != s[j]:
            return -1 if s[i] > s[j] else 1
        return -1 if i < j else 1
    order = sorted(range(len(s)), key=functools.cmp_to_key(cmp))[:k]
    ex = [math.exp(float(s[i]) - float(s[order[0]])) for i in order]
    tot = sum(ex)
    return order, [v / tot for v in ex]


def _brute_dense(x, scores, w1v, w2v, s1, s2, k, quant):
    """y_t = sum_e gate_e(t) FFN_e(x_t) over every expert, gate 0 when unselected."""
    T, H = x.shape
    E, twoI, _ = w1v.shape
    I = twoI // 2
    gates = np.zeros((T, E))
    for t in range(T):
        order, wts = _brute_route(scores[t], k)
        for e, wv in zip(order, wts):
            gates[t, e] = np.float32(wv)
    xv = x.float().numpy()
    if quant == M.FP8_TENSOR:
        sx = np.float32(np.abs(xv).max()) / np.float32(448.0)
        xin = _t_e4m3(xv / sx).astype(np.float64)
    elif quant == M.FP8_BLOCK:
        sxg = np.stack([np.abs(xv[:, g * 128:(g + 1) * 128]).max(axis=1) for g in range(H // 128)], 1)
        sxg = sxg.astype(np.float32) / np.float32(448.0)
        xin = _t_e4m3(xv / np.repeat(sxg, 128, axis=1)).astype(np.float64)
    else:
        xin = xv.astype(np.float64)
    acts = {}
    for t in range(T):
        for e in range(E):
            if gates[t, e] == 0:
                continue
            g = np.zeros(I)
            u = np.zeros(I)
            for i in range(I):
                for G in range(H // 128 if quant == M.FP8_BLOCK else 1):
                    hs = slice(G * 128, (G + 1) * 128) if quant == M.FP8_BLOCK else slice(0, H)
                    dg = float(np.dot(xin[t, hs], w1v[e, i, hs]))
                    du = float(np.dot(xin[t, hs], w1v[e, I + i, hs]))
                    if quant == M.FP8_TENSOR:
                        sc = np.float64(sx) * np.float64(s1[e])
                        dg, du = sc * dg, sc * du
                    elif quant == M.FP8_BLOCK:
                        dg *= np.float64(sxg[t, G]) * np.float64(s1[e, i // 128, G])
                        du *= np.float64(sxg[t, G]) * np.float64(s1[e, (I + i) // 128, G])
                    g[i] += dg
                    u[i] += du
            acts[(t, e)] = _silu_u(g, u).astype(np.float32)
    if quant == M.FP8_TENSOR:
        sh = np.float32(max(np.abs(v).max() for v in acts.values())) / np.float32(448.0)
    y = np.zeros((T, H))
    for (t, e), a in acts.items():
        if quant == M.BF16:
            h = _t_bf16_val(a).astype(np.float64)
            o = w2v[e] @ h
        elif quant == M.FP8_TENSOR:
            h = _t_e4m3(a / sh).astype(np.float64)
            o = (np.float64(sh) * np.float64(s2[e])) * (w2v[e] @ h)
        else:
            o = np.zeros(H)
            for G in range(I // 128):
                seg = a[G * 128:(G + 1) * 128]
                shg = np.float32(np.abs(seg).max()) / np.float32(448.0)
                hq = _t_e4m3(seg / shg).astype(np.float64)
                for c in range(H):
                    o[c] += np.float64(shg) * np.float64(s2[e, c // 128, G]) * float(np.dot(hq, w2v[e, c, G * 128:(G + 1) * 128]))
        y[t] += gates[t, e] * o
    return _t_bf16_val(y)


@pytest.mark.parametrize("quant", [M.BF16, M.FP8_TENSOR, M.FP8_BLOCK])
def test_brute_force_dense_sum_over_all_experts(quant):
    rng = np.random.default_rng(9)
    T, E, k = 3, 4, 2
    H, I = (256, 128)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    scores = rng.standard_normal((T, E)).astype(np.float32)
    w1f = rng.standard_normal((E, 2 * I, H)) / math.sqrt(H)
    w2f = rng.standard_normal((E, H, I)) / math.sqrt(I)
    if quant == M.BF16:
        w1t = torch.from_numpy(w1f).float().to(torch.bfloat16)
        w2t = torch.from_numpy(w2f).float().to(torch.bfloat16)
        w1n, w2n, s1, s2 = bits16(w1t), bits16(w2t), None, None
        w1v, w2v = w1t.double().numpy(), w2t.double().numpy()
    else:
        s1 = (np.abs(w1f).max(axis=(1, 2)) / 448.0).astype(np.float32) if quant == M.FP8_TENSOR else \
            (2.0 ** rng.integers(-9, -6, size=(E, 2 * I // 128, H // 128))).astype(np.float32)
        s2 = (np.abs(w2f).max(axis=(1, 2)) / 448.0).astype(np.float32) if quant == M.FP8_TENSOR else \
            (2.0 ** rng.integers(-9, -6, size=(E, H // 128, I // 128))).astype(np.float32)
        if quant == M.FP8_TENSOR:
            d1 = w1f / s1[:, None, None]
            d2 = w2f / s2[:, None, None]
        else:
            d1 = w1f / np.repeat(np.repeat(s1, 128, 1), 128, 2)
            d2 = w2f / np.repeat(np.repeat(s2, 128, 1), 128, 2)
        q1 = torch.from_numpy(np.clip(d1, -448, 448)).float().to(E4)
        q2 = torch.from_numpy(np.clip(d2, -448, 448)).float().to(E4)
        w1n, w2n = q1.view(torch.uint8).numpy(), q2.view(torch.uint8).numpy()
        w1v, w2v = q1.double().numpy(), q2.double().numpy()
    out = M.forward(bits16(x), scores, w1n, w2n, s1, s2, k, quant)
    ref = _brute_dense(x, scores, w1v, w2v, s1, s2, k, quant)
    ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(out["y"] - ref) <= ulp)
    assert np.mean(out["y"] == ref) > 0.97


@pytest.mark.parametrize("quant", [M.FP8_TENSOR, M.FP8_BLOCK])
def test_fp8_quantisation_noise_is_percent_level(quant):
    import workloads as W
    from tests._util import oracle_args

    wl = W.Workload("noise", 4, 16, 4, 512, 256, quant, 77)
    inp = W.make_inputs(wl)
    x, scores, w1, w2, s1, s2 = oracle_args(inp)
    out = M.forward(x, scores, w1, w2, s1, s2, wl.k, quant)
    # the same forward with unquantised activations and the dequantised weights
    from oracle.formats import e4m3_decode, f32_from_bf16_bits

    if quant == M.FP8_TENSOR:
        W1 = e4m3_decode(w1) * s1[:, None, None]
        W2 = e4m3_decode(w2) * s2[:, None, None]
    else:
        W1 = e4m3_decode(w1) * np.repeat(np.repeat(s1, 128, 1), 128, 2)
        W2 = e4m3_decode(w2) * np.repeat(np.repeat(s2, 128, 1), 128, 2)
    xv = f32_from_bf16_bits(x).astype(np.float64)
    y = np.zeros((wl.T, wl.H))
    for t in range(wl.T):
        for j in range(wl.k):
            e = out["ids"][t, j]
            g = W1[e, :wl.I] @ xv[t]
            u = W1[e, wl.I:] @ xv[t]
            y[t] += out["w"][t, j] * (W2[e] @ (g / (1 + np.exp(-g)) * u))
    err = rel_l2(out["y"], y)
    assert 1e-3 < err < 5e-2


@pytest.mark.parametrize("quant", [M.BF16, M.FP8_TENSOR, M.FP8_BLOCK])
def test_token_subset_gives_exactly_those_rows_of_the_full_forward(quant):
    """forward(tokens=S) is what the full-size GPU parity tests, the CPU baseline
    and the reference arm call: it must return rows S of the full forward bit for
    bit.  The subset skips other tokens' routes, except that the per-tensor scale
    of h still spans every route: the test checks that the subset's own routes
    would give a different amax here, so a scale taken over the subset alone
    would fail it."""
    import workloads as W
    from tests._util import oracle_args

    wl = W.Workload("subset", 40, 16, 4, 256, 256, quant, 88)
    args = oracle_args(W.make_inputs(wl))
    full = M.forward(*args, wl.k, quant)
    S = np.array([0, 3, 4, 17, 39])
    sub = M.forward(*args, wl.k, quant, tokens=S)
    assert np.array_equal(sub["y"].view(np.uint32), full["y"][S].view(np.uint32))
    assert np.array_equal(sub["tokens"], S)
    routes = (S[:, None] * wl.k + np.arange(wl.k)[None, :]).ravel()
    assert np.array_equal(sub["a"][routes].view(np.uint32), full["a"][routes].view(np.uint32))
    if quant == M.FP8_TENSOR:
        assert np.abs(full["a"][routes]).max() < np.abs(full["a"]).max()
    else:  # other tokens' routes were skipped
        others = np.setdiff1d(np.arange(wl.T * wl.k), routes)
        assert np.all(np.isnan(sub["a"][others]))


# ----------------------------------------------------------------------------- shared experts, fp32 partials
def _zero_routed(quant, E, H, I):
    """Routed experts whose weights are all zero: their routes add exactly 0."""
    if quant == M.BF16:
        return np.zeros((E, 2 * I, H), np.uint16), np.zeros((E, H, I), np.uint16), None, None
    w1 = np.zeros((E, 2 * I, H), np.uint8)
    w2 = np.zeros((E, H, I), np.uint8)
    if quant == M.FP8_TENSOR:
        return w1, w2, np.ones(E, np.float32), np.ones(E, np.float32)
    return (w1, w2, np.ones((E, 2 * I // 128, H // 128), np.float32),
            np.ones((E, H // 128, I // 128), np.float32))


@pytest.mark.parametrize("quant", [M.BF16, M.FP8_TENSOR, M.FP8_BLOCK])
def test_shared_identity_expert_closed_form(quant):
    """A shared expert that is identity-like (one nonzero per row, as in the
    routed closed form above) next to routed experts that contribute nothing:
    y must be the SwiGLU closed form of the shared expert alone, for every
    token (weight 1), in all three modes.  A shared expert that were skipped,
    weighted by a routing weight, or read with the routed experts' scales would
    fail it (the routed scales here are 1, the shared ones are not)."""
    c = _identity_case(quant, E=1)
    Er, k = 6, 2
    rng = np.random.default_rng(3)
    w1, w2, s1, s2 = _zero_routed(quant, Er, c["H"], c["I"])
    scores = rng.standard_normal((c["T"], Er)).astype(np.float32)
    shared = {"w1": c["w1"], "w2": c["w2"], "w1_scale": c["s1"], "w2_scale": c["s2"]}
    out = M.forward(bits16(c["x"]), scores, w1, w2, s1, s2, k, quant, shared=shared)
    assert np.array_equal(out["y"], _expected_identity(c, quant))


def test_shared_expert_adds_a_dense_swiglu_to_the_routed_sum():
    """bf16: forward with one shared expert = the routed-only forward's unrounded
    y plus the shared expert's dense SwiGLU MLP (torch CPU, h rounded to bf16),
    rounded once; checked to within one bf16 step (the two sides round the
    routed sum at different points) and equal for nearly every element."""
    rng = np.random.default_rng(11)
    T, E, k, H, I = 12, 5, 2, 256, 128
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    scores = rng.standard_normal((T, E)).astype(np.float32)
    mk = lambda *shape, fan: (torch.from_numpy(rng.standard_normal(shape).astype(np.float32)) / math.sqrt(fan)).to(torch.bfloat16)
    w1, w2 = mk(E, 2 * I, H, fan=H), mk(E, H, I, fan=I)
    s1, s2 = mk(1, 2 * I, H, fan=H), mk(1, H, I, fan=I)
    routed = M.forward(bits16(x), scores, bits16(w1), bits16(w2), None, None, k, M.BF16, y_fp32=True)["y"]
    both = M.forward(bits16(x), scores, bits16(w1), bits16(w2), None, None, k, M.BF16,
                     shared={"w1": bits16(s1), "w2": bits16(s2), "w1_scale": None, "w2_scale": None})["y"]
    X = x.double()
    g = X @ s1[0, :I].double().T
    u = X @ s1[0, I:].double().T
    hh = (Fnn.silu(g) * u).float().to(torch.bfloat16).double()
    dense = (hh @ s2[0].double().T).numpy()
    ref = _t_bf16_val(routed.astype(np.float64) + dense)
    ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(both - ref) <= ulp)
    assert np.mean(both == ref) > 0.99
    assert not np.array_equal(both, _t_bf16_val(routed))  # the shared term is not negligible


@pytest.mark.parametrize("quant", [M.BF16, M.FP8_TENSOR, M.FP8_BLOCK])
def test_fp32_partial_rounds_to_the_bf16_output(quant):
    import workloads as W
    from tests._util import oracle_args

    wl = W.Workload("partial", 10, 8, 2, 256, 256, quant, 90)
    args = oracle_args(W.make_inputs(wl))
    y32 = M.forward(*args, wl.k, quant, y_fp32=True)["y"]
    y16 = M.forward(*args, wl.k, quant)["y"]
    assert np.array_equal(bf16_round_t(y32), y16)
    assert not np.array_equal(y32, y16)  # the partial is not rounded


def bf16_round_t(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).float().numpy()


def tp_slice(w1, w2, s1, s2, quant, P, p):
    """Slice p of P of a tensor-parallel split of the intermediate dimension I:
    gate rows and up rows [p I/P, (p+1) I/P) of W1, the same columns of W2 (and
    the matching 128 x 128 scale blocks)."""
    I = w1.shape[1] // 2
    n = I // P
    rows = np.concatenate([np.arange(p * n, (p + 1) * n), I + np.arange(p * n, (p + 1) * n)])
    w1p, w2p = w1[:, rows], w2[:, :, p * n:(p + 1) * n]
    if quant == M.FP8_BLOCK:
        assert n % 128 == 0
        b = n // 128
        brows = np.concatenate([np.arange(p * b, (p + 1) * b), I // 128 + np.arange(p * b, (p + 1) * b)])
        return w1p, w2p, s1[:, brows], s2[:, :, p * b:(p + 1) * b]
    return w1p, w2p, s1, s2


@pytest.mark.parametrize("quant", [M.BF16, M.FP8_BLOCK])
def test_tensor_parallel_slices_sum_to_the_whole(quant):
    """Splitting I into slices (the TP8 deployment of the route-MMA page's
    Performance section) and summing the slices' unrounded partial outputs gives
    the unsplit forward's unrounded output: every h value and its quantisation
    (bf16, or per 128-column group when the slices are whole groups) is the same
    on both sides, so they differ only by fp32 summation order.  With shared
    experts too (sliced the same way)."""
    import workloads as W
    from tests._util import oracle_args

    wl = W.Workload("tp", 9, 8, 2, 256, 256, quant, 91)
    x, scores, w1, w2, s1, s2 = oracle_args(W.make_inputs(wl))
    sh = oracle_args(W.make_inputs(W.Workload("tp_sh", 9, 1, 1, 256, 256, quant, 92)))
    shared = {"w1": sh[2], "w2": sh[3], "w1_scale": sh[4], "w2_scale": sh[5]}
    whole = M.forward(x, scores, w1, w2, s1, s2, wl.k, quant, shared=shared, y_fp32=True)["y"]
    P = 2
    total = np.zeros_like(whole, dtype=np.float64)
    for p in range(P):
        a1, a2, b1, b2 = tp_slice(w1, w2, s1, s2, quant, P, p)
        c1, c2, d1, d2 = tp_slice(shared["w1"], shared["w2"], shared["w1_scale"], shared["w2_scale"], quant, P, p)
        part = M.forward(x, scores, a1, a2, b1, b2, wl.k, quant, y_fp32=True,
                         shared={"w1": c1, "w2": c2, "w1_scale": d1, "w2_scale": d2})["y"]
        assert np.abs(part).max() > 0.05 * np.abs(whole).max()  # each slice contributes
        total += part
    assert np.max(np.abs(total - whole)) <= 1e-5 * np.abs(whole).max()


# ----------------------------------------------------------------------------- MXFP8
def _mx_torch(v32):
    """MX quantisation written with torch: per run of 32 along the last axis, X =
    (frexp exponent of the run's amax) - 1 - 8 (-127 for a zero run, clamped),
    codes by torch's float8 conversion after a clamp to +-448.  Returns the
    dequantised values (fp64) and the exponents."""
    t = torch.from_numpy(np.asarray(v32, np.float32))
    rows, cols = t.shape
    runs = t.view(rows, cols // 32, 32)
    amax = runs.abs().amax(dim=2)
    _, ex = torch.frexp(amax)
    X = torch.where(amax > 0, ex.long() - 9, torch.full_like(ex.long(), -127)).clamp(-127, 127)
    sc = torch.exp2(X.double())
    q = (runs.double() / sc[..., None]).float().clamp(-448, 448).to(E4).double()
    return (q * sc[..., None]).reshape(rows, cols).numpy(), X.numpy()


def test_mx_identity_experts_closed_form():
    """MXFP8 forward with identity-like experts (one nonzero e4m3 code per weight
    row, random power-of-two run scales), top_k = 1: every dot product has one
    term, so y follows from the SwiGLU formula with x and h quantised per run of
    32 (computed here with torch's float8 conversion and frexp)."""
    rng = np.random.default_rng(12)
    T, E, H, I = 20, 3, 256, 128
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    scores = rng.standard_normal((T, E)).astype(np.float32)
    sig = [rng.permutation(H)[:I] for _ in range(E)]
    pi = [rng.permutation(I) for _ in range(E)]
    w1 = np.zeros((E, 2 * I, H), np.uint8)
    w2 = np.zeros((E, H, I), np.uint8)
    s1 = (127 + rng.integers(-3, 4, size=(E, 2 * I, H // 32))).astype(np.uint8)
    s2 = (127 + rng.integers(-3, 4, size=(E, H, I // 32))).astype(np.uint8)
    for e in range(E):
        w1[e, np.arange(I), sig[e]] = CODE_2
        w1[e, I + np.arange(I), sig[e]] = CODE_1
        w2[e, np.arange(H), pi[e][np.arange(H) % I]] = CODE_1
    out = M.forward(bits16(x), scores, w1, w2, s1, s2, 1, M.MXFP8)
    xq, _ = _mx_torch(x.float().numpy())
    e_of = np.argmax(scores, axis=1)
    a = np.zeros((T, I), np.float32)
    for t in range(T):
        e = e_of[t]
        s = sig[e]
        i = np.arange(I)
        g = 2.0 * xq[t, s] * np.exp2(s1[e, i, s // 32].astype(np.float64) - 127)
        u = xq[t, s] * np.exp2(s1[e, I + i, s // 32].astype(np.float64) - 127)
        a[t] = _silu_u(g, u)
    hq, _ = _mx_torch(a)
    y = np.zeros((T, H))
    for t in range(T):
        e = e_of[t]
        src = pi[e][np.arange(H) % I]
        y[t] = hq[t, src] * np.exp2(s2[e, np.arange(H), src // 32].astype(np.float64) - 127)
    assert np.array_equal(out["y"], _t_bf16_val(y))


def test_mx_brute_force_dense_sum_over_all_experts():
    rng = np.random.default_rng(13)
    T, E, k, H, I = 3, 4, 2, 128, 64
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    scores = rng.standard_normal((T, E)).astype(np.float32)
    import workloads as W

    w1c, s1 = W._pack_mxfp8(torch.from_numpy(rng.standard_normal((E, 2 * I, H)) / math.sqrt(H)).float())
    w2c, s2 = W._pack_mxfp8(torch.from_numpy(rng.standard_normal((E, H, I)) / math.sqrt(I)).float())
    w1v = w1c.view(E4).double() * torch.exp2(s1.double() - 127).repeat_interleave(32, dim=2)
    w2v = w2c.view(E4).double() * torch.exp2(s2.double() - 127).repeat_interleave(32, dim=2)
    out = M.forward(bits16(x), scores, w1c.numpy(), w2c.numpy(), s1.numpy(), s2.numpy(), k, M.MXFP8)
    xin, _ = _mx_torch(x.float().numpy())
    y = np.zeros((T, H))
    for t in range(T):
        order, wts = _brute_route(scores[t], k)
        for e, wv in zip(order, wts):
            g = w1v[e, :I].numpy() @ xin[t]
            u = w1v[e, I:].numpy() @ xin[t]
            a = _silu_u(g, u).astype(np.float32)[None, :]
            h, _ = _mx_torch(a)
            y[t] += np.float32(wv) * (w2v[e].numpy() @ h[0])
    ref = _t_bf16_val(y)
    assert np.all(np.abs(out["y"] - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)
    assert np.mean(out["y"] == ref) > 0.97


def test_mx_quantisation_noise_is_percent_level():
    import workloads as W
    from oracle.mx import mx_dequantize
    from tests._util import oracle_args

    wl = W.Workload("mxnoise", 4, 16, 4, 512, 256, W.QUANT_MXFP8, 78)
    x, scores, w1, w2, s1, s2 = oracle_args(W.make_inputs(wl))
    out = M.forward(x, scores, w1, w2, s1, s2, wl.k, M.MXFP8)
    from oracle.formats import f32_from_bf16_bits

    xv = f32_from_bf16_bits(x).astype(np.float64)
    y = np.zeros((wl.T, wl.H))
    for t in range(wl.T):
        for j in range(wl.k):
            e = out["ids"][t, j]
            W1 = mx_dequantize(w1[e], s1[e])
            g, u = W1[:wl.I] @ xv[t], W1[wl.I:] @ xv[t]
            y[t] += out["w"][t, j] * (mx_dequantize(w2[e], s2[e]) @ (g / (1 + np.exp(-g)) * u))
    err = rel_l2(out["y"], y)
    # larger than the fp32-scaled forms: the OCP shared exponent floor(log2 amax) - 8
    # leaves amax / 2^X in [256, 512), so a run whose amax has a significand of 1.75 or
    # more (about a fifth of runs) saturates its largest values at 448, by up to 12.5%
    assert 1e-3 < err < 1e-1
