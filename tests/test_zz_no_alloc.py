"""moe_shuffle_noalloc: the shuffle entry point that allocates nothing.

It is meant for callers that cannot allocate device memory when they need the
shuffle (inside a CUDA-graph capture, plugins of a framework that owns all
device memory, serving loops with a fixed footprint); its scratch is a fixed
array inside the library.  Its results must equal those of moe_shuffle (which
takes a caller workspace), bit for bit, call after call: the shared array keeps
the previous call's contents, so two different calls in a row are checked.

This file is collected last so that a run stopping at the first failure has run
every other test before it; it also passes on its own in a fresh process."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def m():
    import __graft_entry__

    __graft_entry__.build()
    import mixture_experts_layer_index_gb300 as mod

    return mod


def _ids(seed, T, E, k):
    rng = np.random.default_rng(seed)
    keys = rng.random((T, E)) ** np.linspace(1.0, 6.0, E)[None, :]  # skewed popularity
    return np.argsort(-keys, axis=1)[:, :k].astype(np.int32)


def _outputs(T, E, k):
    R = T * k
    return (torch.full((E,), -1, dtype=torch.int32, device=DEV),
            torch.full((E + 1,), -1, dtype=torch.int32, device=DEV),
            torch.full((R,), -1, dtype=torch.int32, device=DEV),
            torch.full((R,), -1, dtype=torch.int32, device=DEV))


def _with_workspace(m, ids, T, E, k):
    out = _outputs(T, E, k)
    ws = torch.empty(m.moe_shuffle_workspace_size(T, E, k), dtype=torch.uint8, device=DEV)
    m.moe_shuffle(ids, T, E, k, *out, ws)
    return out


def _without_workspace(m, ids, T, E, k):
    out = _outputs(T, E, k)
    m.moe_shuffle_noalloc(ids, T, E, k, *out)
    return out


def test_noalloc_matches_workspace_shuffle_on_consecutive_calls(m):
    cases = [(16384, 128, 8, 1), (37, 16, 3, 2), (2048, 64, 8, 3)]  # a big call, then smaller ones
    for T, E, k, seed in cases:
        ids = torch.from_numpy(_ids(seed, T, E, k)).to(DEV)
        ref = _with_workspace(m, ids, T, E, k)
        got = _without_workspace(m, ids, T, E, k)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_noalloc_rejects_problems_beyond_its_fixed_scratch(m):
    T, E, k = 40000, 128, 8  # 320000 routes: more scratch than the fixed array holds
    assert m.moe_shuffle_workspace_size(T, E, k) > (1 << 20)
    ids = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    out = _outputs(T, E, k)
    with pytest.raises(m.MoeError) as ei:
        m.moe_shuffle_noalloc(ids, T, E, k, *out)
    assert ei.value.status == m.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out[0] == -1)  # nothing was launched
