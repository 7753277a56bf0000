"""CPU oracle for the fused norm + feed-forward block.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 statement of what the block
computes, written from the TransformerEngine JAX pages (Activation, LayerNorm MLP, LayerNorm
Dense).  Only the test suite, the package's smoke check and the benchmark's CPU-baseline leg
may import it.  The CUDA library never calls it, shares no code with it, and has no fallback
to it.

Modules:
  numerics  fp32 / bf16 / E4M3 rounding and per-tensor scaling, from the formats' definitions
  block     normalization, activations, GEMM + bias, the composed forward and backward passes

Every function is pinned by tests under ``tests/test_oracle_*.py`` against something other
than itself: library routines (torch's layer_norm / rms_norm / autograd / float8 and bfloat16
conversions, scipy's erf), closed forms, identities, brute force and finite differences.
"""

from . import block, numerics  # noqa: F401
