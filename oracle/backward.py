"""The input gradient of the linear layer, and the whole layer backward with its ordering.

TEST INFRASTRUCTURE ONLY (see the package docstring).

FORGE summary, §5 Significance and claims, limitations: the fused update may run
only after the layer's input gradient has been read from the weights, because
the update overwrites them.  For the linear layer Y = X W^T the input gradient
is dX = dY W, with dY [T, d_out] and W [d_out, d_in]: it needs the weights as
they were BEFORE the step.  The layer backward is therefore, in this order:

  1. dX = dY W_old, summed exactly (float64: bf16 x bf16 products are exact, and a
     float64 sum of d_out <= 2^16 of them is far inside one binary32 ULP of the
     result), rounded once to binary32 and then once, to nearest even, to
     bfloat16 -- the activation-gradient format of dY and X (§2 Precision and
     fidelity: activations and their gradients are BF16);
  2. the fused weight step of ``step.fused_step`` on dW = dY^T X.

dX[t, i] = sum_o dY[t, o] W[o, i].  Layout: dX [T, d_in] row-major bfloat16 bits.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from . import bf16, step

_CHUNK = 1 << 22


def dx_f32(dy_bits, w_bits) -> np.ndarray:
    """dY W in binary32 [T, d_in] (the sum exact in float64, one rounding)."""
    dy = bf16.to_f64(dy_bits)
    w = bf16.to_f64(w_bits)
    return (dy @ w).astype(np.float32)


def dx(dy_bits, w_bits) -> np.ndarray:
    """dX = dY W as bfloat16 bits [T, d_in]: binary32, then round-to-nearest-even."""
    return bf16.round_nearest_even(dx_f32(dy_bits, w_bits))


def dx_at(dy_bits, w_bits, rows: Sequence[int], cols: Sequence[int]) -> Dict[str, np.ndarray]:
    """dX at listed (token, column) positions, one d_out-term dot product each.

    Returns the binary32 values (``f32``) and their bfloat16 bits (``bits``)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    d_out = np.asarray(w_bits).shape[0]
    out = np.empty(rows.shape[0], dtype=np.float32)
    n = max(1, _CHUNK // max(d_out, 1))
    for s in range(0, rows.shape[0], n):
        r, c = rows[s:s + n], cols[s:s + n]
        a = bf16.to_f64(np.asarray(dy_bits)[r, :])
        b = bf16.to_f64(np.asarray(w_bits)[:, c]).T
        out[s:s + n] = np.einsum("nk,nk->n", a, b).astype(np.float32)
    return {"f32": out, "bits": bf16.round_nearest_even(out)}


def linear_backward(opt: str, dy_bits, x_bits, w_bits, m, v, hp, t: int, seed: int,
                    state: str = "fp32", m_scales=None, v_scales=None) -> Dict[str, Optional[np.ndarray]]:
    """dX from the weights before the step, then the fused weight step.

    Returns the fused step's outputs (W, w_f32, m, v, scales, g) plus dX (bits) and dx_f32."""
    d32 = dx_f32(dy_bits, w_bits)           # step 1 reads W_old ...
    out = step.fused_step(opt, dy_bits, x_bits, w_bits, m, v, hp, t, seed, state, m_scales, v_scales)  # ... step 2 replaces it
    out["dX"] = bf16.round_nearest_even(d32)
    out["dx_f32"] = d32
    return out
