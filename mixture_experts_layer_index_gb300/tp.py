"""Tensor-parallel split of the intermediate dimension I across ranks.

The route-MMA page ("perf: add small-batch route MMA for MoE", Performance)
measures its per-tensor FP8 shape as one rank of an eight-way tensor-parallel
deployment ("Hunyuan-V3 TP8": E=192, H=4096, I=192 per rank).  Under that
split, rank p of P holds gate rows and up rows [p*I/P, (p+1)*I/P) of every
W1[e] and the same columns of every W2[e]; it runs the whole routed forward on
its slice (routing and x are replicated), producing an unrounded partial y;
the partials are summed across ranks and the sum is rounded once.

This module is argument marshalling and the collective only: the slicing is
indexing of the caller's tensors, the sum is torch.distributed.all_reduce
(NCCL between GPUs), and every arithmetic step of the forward and the final
rounding runs in the library's kernels (moe_forward_ex with y_fp32 = 1, then
moe_round_bf16).
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import (MOE_BF16, MOE_FP8_BLOCK128, QUANT_BY_NAME, forward_options, moe_forward_ex, moe_round_bf16,
               problem)


def _quant_code(quant) -> int:
    return QUANT_BY_NAME[quant] if isinstance(quant, str) else int(quant)


def shard_weights(w1: torch.Tensor, w2: torch.Tensor, w1_scale: Optional[torch.Tensor],
                  w2_scale: Optional[torch.Tensor], quant, rank: int, world: int) -> Tuple:
    """Slice `rank` of `world` of the expert weights W1 [E, 2I, H], W2 [E, H, I]
    (and their scales): gate rows and up rows [rank*I/world, (rank+1)*I/world)
    of W1, the same columns of W2; for 128x128-blockwise FP8 the matching scale
    blocks, so I/world must be a multiple of 128 there.  Per-tensor scales are
    kept whole (each slice's codes keep their matrix's scale).  Returns
    contiguous (w1, w2, w1_scale, w2_scale) for the slice."""
    q = _quant_code(quant)
    I = w1.shape[1] // 2
    if I % world:
        raise ValueError(f"I = {I} does not split into {world} slices")
    n = I // world
    idx = torch.cat([torch.arange(rank * n, (rank + 1) * n), I + torch.arange(rank * n, (rank + 1) * n)])
    idx = idx.to(w1.device)
    w1r = w1.index_select(1, idx).contiguous()
    w2r = w2[:, :, rank * n:(rank + 1) * n].contiguous()
    s1r, s2r = w1_scale, w2_scale
    if q == MOE_FP8_BLOCK128:
        if n % 128:
            raise ValueError("blockwise FP8 slices must hold whole 128-column scale groups")
        b = n // 128
        bidx = torch.cat([torch.arange(rank * b, (rank + 1) * b), I // 128 + torch.arange(rank * b, (rank + 1) * b)])
        s1r = w1_scale.index_select(1, bidx.to(w1_scale.device)).contiguous()
        s2r = w2_scale[:, :, rank * b:(rank + 1) * b].contiguous()
    elif q != MOE_BF16:
        s1r, s2r = w1_scale.contiguous(), w2_scale.contiguous()
    return w1r, w2r, s1r, s2r


def allreduce_partial(y32: torch.Tensor, group=None) -> torch.Tensor:
    """Sum the ranks' fp32 partial outputs in place (torch.distributed)."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(y32, op=dist.ReduceOp.SUM, group=group)
    return y32


def forward(T: int, E: int, k: int, H: int, I_slice: int, quant, x, scores, w1, w2, w1_scale, w2_scale,
            y: torch.Tensor, y32: torch.Tensor, ws: torch.Tensor, shared=None, group=None, stream=None) -> None:
    """This rank's part of a tensor-parallel forward: the routed forward on the
    rank's weight slice (I_slice = I / world columns) with an unrounded fp32
    output, the sum over ranks, and the single rounding of the sum into y.
    `shared` optionally holds this rank's slice of the shared experts as
    (n_shared, w1, w2, w1_scale, w2_scale).  ws must hold moe_workspace_size_ex
    bytes for the slice's problem."""
    p = problem(T, E, k, H, I_slice, quant)
    opt = forward_options(*(shared or (0, None, None, None, None)), y_fp32=True)
    moe_forward_ex(p, opt, x, scores, w1, w2, w1_scale, w2_scale, y32, ws, stream=stream)
    allreduce_partial(y32, group)
    moe_round_bf16(y32, y, stream=stream)
