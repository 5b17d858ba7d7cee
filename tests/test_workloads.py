"""Seeded input generators: determinism, shapes, and the skewed-routing recipe."""
import numpy as np
import torch

import workloads as W
from oracle import moe as M


def test_generators_are_deterministic():
    a = W.make_inputs(W.workload("tiny"))
    b = W.make_inputs(W.workload("tiny"))
    for key in ("x", "scores", "w1", "w2"):
        assert torch.equal(a[key], b[key])


def test_decode_sweep_shares_weights_across_batch():
    h3, h5 = W.workload("hunyuan", 3), W.workload("hunyuan", 5)
    assert h3.weight_seed == h5.weight_seed and h3.seed != h5.seed
    small = W.Workload("s", 4, 6, 2, 128, 64, W.QUANT_FP8_TENSOR, 9)
    w3 = W.make_weights(small.with_tokens(3))
    w5 = W.make_weights(small.with_tokens(5))
    assert torch.equal(w3[0], w5[0]) and torch.equal(w3[2], w5[2])


def test_fp8_weights_fit_their_scales():
    wl = W.Workload("q", 1, 4, 2, 256, 128, W.QUANT_FP8_BLOCK, 5)
    q1, _, s1, _ = W.make_weights(wl)
    assert q1.dtype == torch.uint8 and s1.shape == (4, 2, 2)
    vals = q1.view(torch.float8_e4m3fn).float()
    assert torch.isfinite(vals).all() and vals.abs().max() <= 448


def test_prefill_skew_leaves_four_experts_empty():
    wl = W.workload("prefill")
    ids, _ = M.route(W.make_scores(wl).numpy(), wl.k)
    counts = np.bincount(ids.ravel(), minlength=wl.E)
    assert (counts == 0).sum() == 4
    assert counts.max() <= wl.T
    # Zipf-like: the most popular expert is far above the uniform share
    assert counts.max() > 10 * wl.R / wl.E
