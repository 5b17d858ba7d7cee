"""Tensor-parallel split of I across two ranks, run as two gloo processes on the
CPU: each rank slices the weights with the library's shard_weights, computes its
slice's unrounded partial output (here with the CPU oracle, since there is no GPU
in this test), and the partials are summed with the library's allreduce_partial.
The sum must equal the unsplit forward's unrounded output up to fp32 summation
order, and its single rounding the unsplit bf16 output up to one bf16 step, in
bf16 and blockwise FP8 (whole 128-column groups per slice), with a shared
expert sliced the same way.  The GPU side of each rank (moe_forward_ex with
y_fp32 and moe_round_bf16) is covered by the GPU parity tests."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(quant):
    import workloads as W

    wl = W.Workload(f"tpg_{quant}", 7, 8, 2, 256, 256, quant, 95)
    sh = W.Workload(f"tpg_{quant}_sh", 7, 1, 1, 256, 256, quant, 96)
    return wl, W.make_inputs(wl), W.make_weights(sh)


def _np(t):
    from tests._util import bits16, u8

    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return bits16(t)
    if t.dtype == torch.uint8:
        return u8(t)
    return t.numpy()


def _worker(rank, world, port, quant, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from mixture_experts_layer_index_gb300 import tp
        from oracle import moe as O

        wl, inp, shw = _case(quant)
        w1, w2, s1, s2 = tp.shard_weights(inp["w1"], inp["w2"], inp["w1_scale"], inp["w2_scale"], quant, rank, world)
        c1, c2, d1, d2 = tp.shard_weights(*shw, quant, rank, world)
        part = O.forward(_np(inp["x"]), inp["scores"].numpy(), _np(w1), _np(w2), _np(s1), _np(s2), wl.k, quant,
                         shared={"w1": _np(c1), "w2": _np(c2), "w1_scale": _np(d1), "w2_scale": _np(d2)},
                         y_fp32=True)["y"]
        y32 = torch.from_numpy(part.copy())
        tp.allreduce_partial(y32)
        out[rank] = y32.numpy()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("quant", ["bf16", "fp8_block"])
def test_tp_two_ranks_sum_to_the_unsplit_forward(quant):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, quant, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=300)
            assert p.exitcode == 0
        res = dict(out)
    from oracle import moe as O

    wl, inp, shw = _case(quant)
    shared = {"w1": _np(shw[0]), "w2": _np(shw[1]), "w1_scale": _np(shw[2]), "w2_scale": _np(shw[3])}
    args = (_np(inp["x"]), inp["scores"].numpy(), _np(inp["w1"]), _np(inp["w2"]), _np(inp["w1_scale"]),
            _np(inp["w2_scale"]), wl.k, quant)
    whole32 = O.forward(*args, shared=shared, y_fp32=True)["y"]
    whole16 = O.forward(*args, shared=shared)["y"]
    assert np.array_equal(res[0], res[1])  # every rank holds the same sum
    assert np.max(np.abs(res[0] - whole32)) <= 1e-5 * np.abs(whole32).max()
    y = torch.from_numpy(res[0]).to(torch.bfloat16).float().numpy()
    assert np.all(np.abs(y - whole16) <= np.abs(whole16) * 2.0 ** -7 + 1e-30)


def test_shard_weights_rejects_splits_that_break_scale_groups():
    from mixture_experts_layer_index_gb300 import tp

    wl, inp, _ = _case("fp8_block")
    with pytest.raises(ValueError):
        tp.shard_weights(inp["w1"], inp["w2"], inp["w1_scale"], inp["w2_scale"], "fp8_block", 0, 4)  # 64 columns
    with pytest.raises(ValueError):
        tp.shard_weights(inp["w1"], inp["w2"], None, None, "bf16", 0, 3)
