"""CPU oracle for the block-scaled MoE GEMM path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
restatement of what the GPU path computes, written from the definitions on the
pages it cites, in float64 (and in float32 exactly where a rounding decision
turns a float into an integer code, so both sides decide in the same
precision).  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  The product path (the CUDA library and its
Python binding) never imports, links or executes anything in here, and this
package imports nothing from the product path.

Modules
-------
formats  element and scale codecs (E4M3, E2M1, UE8M0, UE4M3) by value table
quant    scale derivation, group-wise quantisation, the 128x4 SfAtom layout
gemm     dequantise-then-float64 GEMM: dense, grouped contiguous, grouped masked
glu      SwiGLU forward + requantisation, dSwiGLU and dGeGLU backward closed forms
permute  routing permute of tokens and scales into the masked-GEMM layout

Every function is pinned by ``tests/test_oracle_*.py`` against something other
than itself (library decoders, hand-worked values, exact rational brute force,
finite differences, invariants).
"""

from . import formats, quant, gemm, glu, permute  # noqa: F401

__all__ = ["formats", "quant", "gemm", "glu", "permute"]
