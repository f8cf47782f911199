"""CPU oracle for the fused weight-gradient + optimizer step.  TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it: no kernels, headers, helpers, tables or constants.

What it computes, and from which passage of "FORGE: Fused On-Register Gradient
Elimination for Memory-Efficient LLM Training" (gist.science technical summary):

* the weight gradient dW = dY^T X of a linear layer, exact in float64 and
  rounded once to float32 (§2 Methodology, Core mechanism, step 1; §2 Precision
  and fidelity, "Exactness": the fused schedule differs from the full-gradient
  step only in the order of the floating-point sum over tokens) -- ``step.py``;
* one of the eight element-wise optimizers named in §3 Key contributions,
  "Generality", written from each optimizer's own published definition in
  float64 (the summary gives no formulas) -- ``optim.py``;
* the stochastic rounding of the weight write-back to bfloat16 (§2 Precision and
  fidelity, "Low-precision fidelity", second point), with its own counter-based
  Philox4x32-10 generator -- ``bf16.py``, ``philox.py``;
* INT8 optimizer states with one absmax scale per 64-element block (§2 Precision
  and fidelity, third point) -- ``int8_block.py``;
* the layer's input gradient dX = dY W from the weights before the step, and the
  layer backward in that order (§5 Significance and claims, limitations: the
  input gradient must be read before the weights are updated) -- ``backward.py``;
* FP8 (E4M3) operands with per-tensor or per-channel scales, dequantised on the
  gradient tile (§4 Experimental results, "Composability") -- ``fp8.py``.

Every function here is pinned by tests under ``tests/`` against closed forms,
textbook or library routines (``torch.optim`` in float64), brute force on tiny
inputs, or a published known-answer value.
"""
from . import backward, bf16, fp8, int8_block, optim, philox, step  # noqa: F401
