"""CPU oracle for the routed Mixture-of-Experts FFN forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its Python binding) never imports, links or executes it,
and this package never imports the product path: the two share no code.

It is a plain, slow, obviously correct restatement of what the method computes,
written in numpy:

  * ``formats``  - bf16 round-to-nearest-even and the OCP FP8 E4M3 format
                   (decode table, round-to-nearest-even with saturation).
  * ``moe``      - top-k routing, index shuffling (counts, offsets, stable
                   permutation, inverse), the GEMM tile map, activation
                   quantisation and the full forward (bf16, per-tensor FP8,
                   128x128-blockwise FP8), and the weighted top-k combine.

The steps follow the expert-grouped pipeline described in the Motivation
section of "perf: add small-batch route MMA for MoE" (group the routes by
expert, gather their rows, build prefix sums and a GEMM task map, run the
Gate/Up grouped GEMM, the activation with optional re-quantisation, the Down
grouped GEMM, and reduce the k expert outputs of each token), and the
index_shuffling / scatter_add_dense_tokens pair of "Port necessary FBGEMM MoE
kernels".  Accumulations run in fp64; every rounding that the method
defines (bf16 h, e4m3 activations, fp32 scales) is applied in fp32 exactly as
stated in the docstrings of ``moe``.

Every function is pinned by CPU tests (``tests/test_oracle_*.py``) against
closed forms, brute force, invariants and library routines; see the module
docstrings for which pin covers which function.
"""
from . import formats, moe  # noqa: F401
