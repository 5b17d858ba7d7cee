"""Seeded synthetic inputs for the routed MoE FFN forward.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It holds no arithmetic of the forward pass itself: it only draws
random tensors and, for the FP8 workloads, packs the drawn weights into the
e4m3 codes + fp32 scales that the forward pass takes as *inputs* (using
torch's own float8 conversion, a library routine).

Workloads (shapes follow the routed-MoE pages: the world-model layer with 16
experts and top-8 routing from "Port necessary FBGEMM MoE kernels", and the
Hunyuan-V3 TP8 / Qwen3 decode shapes of "perf: add small-batch route MMA for
MoE", Performance tables):

  tiny      T=16,    E=8,   k=2, H=256,  I=128,  bf16
  world16   T=4096,  E=16,  k=8, H=1024, I=1024, bf16, uniform load
  hunyuan   B=1..8,  E=192, k=8, H=4096, I=192,  fp8 per-tensor decode
  qwen3a    B=1..8,  E=128, k=8, H=2048, I=768,  fp8 128x128 blockwise decode
  qwen3b    B=1..8,  E=128, k=8, H=4096, I=512,  fp8 128x128 blockwise decode
  prefill   T=16384, E=128, k=8, H=2048, I=768,  bf16, Zipf(1.1)-skewed routing

Distributions: x ~ N(0,1) rounded to bf16; router scores ~ N(0,1) fp32;
W1 ~ N(0, 1/H), W2 ~ N(0, 1/I) (fan-in scaling), rounded to bf16 or packed to
e4m3 with one fp32 scale per expert matrix (per-tensor) or per 128x128 block
(blockwise), scale = amax / 448 (448 = largest finite e4m3).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

QUANT_BF16 = "bf16"
QUANT_FP8_TENSOR = "fp8_tensor"
QUANT_FP8_BLOCK = "fp8_block"
QUANT_MXFP8 = "mxfp8"
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    E: int
    k: int
    H: int
    I: int
    quant: str
    seed: int
    skew: bool = False
    wseed: int = -1  # weight stream seed; -1 = same as seed

    @property
    def weight_seed(self) -> int:
        return self.seed if self.wseed < 0 else self.wseed

    @property
    def R(self) -> int:
        return self.T * self.k

    def with_tokens(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T, name=f"{self.name}_T{T}", wseed=self.weight_seed)


def _base(name):
    return {
        "tiny": Workload("tiny", 16, 8, 2, 256, 128, QUANT_BF16, 1000),
        "world16": Workload("world16", 4096, 16, 8, 1024, 1024, QUANT_BF16, 1001),
        "hunyuan": Workload("hunyuan", 1, 192, 8, 4096, 192, QUANT_FP8_TENSOR, 1002),
        "qwen3a": Workload("qwen3a", 1, 128, 8, 2048, 768, QUANT_FP8_BLOCK, 1003),
        "qwen3b": Workload("qwen3b", 1, 128, 8, 4096, 512, QUANT_FP8_BLOCK, 1003),
        "prefill": Workload("prefill", 16384, 128, 8, 2048, 768, QUANT_BF16, 1004, skew=True),
    }[name]


def workload(name: str, B: Optional[int] = None) -> Workload:
    """Named workload; for the decode sweeps ``B`` (1..8) sets the token count."""
    w = _base(name)
    if B is not None:
        w = dataclasses.replace(w, T=B, name=f"{name}_B{B}", seed=w.seed * 100 + B,
                                wseed=w.weight_seed)
    return w


DECODE_SWEEPS = ("hunyuan", "qwen3a", "qwen3b")


def _gen(seed: int, stream: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + stream)
    return g


def _bf16(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16)


def _pack_e4m3_per_tensor(w: torch.Tensor):
    """w [E, rows, cols] fp32 -> (codes uint8 [E,rows,cols], scale fp32 [E])."""
    amax = w.abs().amax(dim=(1, 2))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).float()
    q = (w / scale[:, None, None]).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).contiguous(), scale.contiguous()


def _pack_e4m3_block128(w: torch.Tensor):
    """w [E, rows, cols] fp32 -> (codes [E,rows,cols], scale [E, ceil(rows/128), ceil(cols/128)])."""
    E, rows, cols = w.shape
    rb, cb = math.ceil(rows / 128), math.ceil(cols / 128)
    pad = torch.zeros(E, rb * 128, cb * 128, dtype=torch.float32, device=w.device)
    pad[:, :rows, :cols] = w
    blk = pad.view(E, rb, 128, cb, 128)
    amax = blk.abs().amax(dim=(2, 4))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).float()
    q = (blk / scale[:, :, None, :, None]).clamp(-E4M3_MAX, E4M3_MAX)
    q = q.view(E, rb * 128, cb * 128)[:, :rows, :cols].contiguous()
    return q.to(torch.float8_e4m3fn).view(torch.uint8).contiguous(), scale.contiguous()


def _pack_mxfp8(w: torch.Tensor):
    """w [E, rows, cols] fp32 (cols a multiple of 32) -> (e4m3 codes [E, rows, cols],
    E8M0 scale codes uint8 [E, rows, cols/32]): each run of 32 values along a row
    shares 2^X with X = (exponent of the run's amax) - 8, saturating codes.  The
    exponent comes from torch.frexp; the codes from torch's float8 conversion."""
    E, rows, cols = w.shape
    runs = w.view(E, rows, cols // 32, 32)
    amax = runs.abs().amax(dim=3)
    _, ex = torch.frexp(amax)
    X = torch.where(amax > 0, ex.long() - 1 - 8, torch.full_like(ex.long(), -127)).clamp(-127, 127)
    q = (runs / torch.exp2(X.double()).float()[..., None]).clamp(-E4M3_MAX, E4M3_MAX)
    codes = q.reshape(E, rows, cols).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return codes, (X + 127).to(torch.uint8).contiguous()


def skew_bias(E: int, seed: int) -> torch.Tensor:
    """Per-expert router bias giving Zipf(s=1.1) popularity: rank r_e (a seeded
    permutation of 1..E) gets bias -1.1*ln(r_e), so exp(bias) = r_e^-1.1; the four
    least popular ranks get -1e4 and therefore receive no tokens at all."""
    g = _gen(seed, 7)
    r = (torch.randperm(E, generator=g) + 1).double()
    bias = -1.1 * torch.log(r)
    bias[r > E - 4] = -1.0e4
    return bias.float()


def make_scores(wl: Workload) -> torch.Tensor:
    s = torch.randn(wl.T, wl.E, generator=_gen(wl.seed, 1), dtype=torch.float32)
    if wl.skew:
        s = s + skew_bias(wl.E, wl.seed)[None, :]
    return s.contiguous()


def make_x(wl: Workload) -> torch.Tensor:
    return _bf16(torch.randn(wl.T, wl.H, generator=_gen(wl.seed, 0))).contiguous()


def make_weights(wl: Workload, device="cpu"):
    """Returns (w1, w2, w1_scale, w2_scale).  bf16: tensors of dtype bfloat16,
    scales None.  FP8: uint8 e4m3 codes plus fp32 scales.  The weight streams
    do not depend on T, so every B of a decode sweep sees the same experts.
    ``device`` selects where the seeded generator draws (a CUDA generator draws
    a different, equally seeded stream than the CPU one)."""
    g1 = _gen(wl.weight_seed, 2, device)
    g2 = _gen(wl.weight_seed, 3, device)
    w1 = torch.randn(wl.E, 2 * wl.I, wl.H, generator=g1, device=device) * (1.0 / math.sqrt(wl.H))
    w2 = torch.randn(wl.E, wl.H, wl.I, generator=g2, device=device) * (1.0 / math.sqrt(wl.I))
    if wl.quant == QUANT_BF16:
        return _bf16(w1).contiguous(), _bf16(w2).contiguous(), None, None
    if wl.quant == QUANT_FP8_TENSOR:
        q1, s1 = _pack_e4m3_per_tensor(w1)
        q2, s2 = _pack_e4m3_per_tensor(w2)
        return q1, q2, s1, s2
    if wl.quant == QUANT_FP8_BLOCK:
        q1, s1 = _pack_e4m3_block128(w1)
        q2, s2 = _pack_e4m3_block128(w2)
        return q1, q2, s1, s2
    if wl.quant == QUANT_MXFP8:
        q1, s1 = _pack_mxfp8(w1)
        q2, s2 = _pack_mxfp8(w2)
        return q1, q2, s1, s2
    raise ValueError(wl.quant)


def make_inputs(wl: Workload):
    """All inputs of one forward call, on the CPU, as a dict of torch tensors."""
    w1, w2, s1, s2 = make_weights(wl)
    return {
        "x": make_x(wl),
        "scores": make_scores(wl),
        "w1": w1,
        "w2": w2,
        "w1_scale": s1,
        "w2_scale": s2,
    }
