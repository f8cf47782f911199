"""The whole fused step: weight gradient, optimizer, state write-back, weight rounding.

FORGE summary, §2 Methodology, Core mechanism: for one weight tile the kernel
(1) accumulates the products of the upstream gradient dY and the input
activation X in FP32, (2) applies the optimizer to the finished tile, (3)
discards the gradient tile, (4) writes back only the updated weight tile and
the (optionally quantised) moment tiles.  §2 Precision and fidelity,
"Exactness": for an element-wise optimizer this equals the ordinary step on the
full gradient up to the order of the sum over tokens.  The oracle therefore
computes the full-gradient step by its plain definition, in this order:

  1. g = binary32( dY^T X ), the sum exact in float64 (bf16 x bf16 products are
     exact in float64; a float64 sum of T <= 2^16 such terms is within
     T * 2^-53 * sum|terms| of exact, far below one binary32 ULP of the result),
     then one round-to-nearest-even to binary32 (§2 Precision and fidelity: the
     gradient is consumed in FP32 and never truncated to BF16);
  2. INT8 states are dequantised (int8_block.dequantize);
  3. the optimizer runs in float64 (optim.update);
  4. new moments are rounded to binary32, or requantised to INT8 with one absmax
     scale per 64-block, or rounded to binary32 and then stochastically to BF16
     with their own Philox streams (§2 Precision and fidelity, "BF16 or INT8"
     states); the weight update itself uses the unrounded moments;
  5. the new weight is rounded to binary32, then stochastically to bfloat16
     with 16 Philox bits keyed by (seed, step, element index) (bf16, philox).

Layouts: dY [T, d_out] and X [T, d_in] row-major bfloat16 bit patterns (uint16);
W [d_out, d_in] bfloat16 bits; m, v [d_out, d_in] binary32, int8 codes or bfloat16 bits; INT8
scales [d_out, d_in / 64] binary32 per moment.  dW[o, i] = sum_t dY[t, o] X[t, i]
is the weight gradient of the linear layer Y = X W^T.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

from . import bf16, int8_block, optim, philox

_CHUNK = 1 << 22  # elements of a gathered T x n block kept in memory at once


def dw(dy_bits, x_bits) -> np.ndarray:
    """Full weight gradient, binary32 [d_out, d_in]."""
    dy = bf16.to_f64(dy_bits)
    x = bf16.to_f64(x_bits)
    return (dy.T @ x).astype(np.float32)


def dw_at(dy_bits, x_bits, rows: Sequence[int], cols: Sequence[int]) -> np.ndarray:
    """dW at the listed (row, col) positions, binary32, computed one position at a time in blocks."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    T = np.asarray(dy_bits).shape[0]
    out = np.empty(rows.shape[0], dtype=np.float32)
    step = max(1, _CHUNK // max(T, 1))
    for s in range(0, rows.shape[0], step):
        r, c = rows[s:s + step], cols[s:s + step]
        a = bf16.to_f64(np.asarray(dy_bits)[:, r])
        b = bf16.to_f64(np.asarray(x_bits)[:, c])
        out[s:s + step] = np.einsum("tn,tn->n", a, b).astype(np.float32)
    return out


def dw_blocks(dy_bits, x_bits, rows: Sequence[int], col0: Sequence[int], width: int = 64) -> np.ndarray:
    """dW over ``width`` consecutive columns starting at each (row, col0): binary32 (n, width)."""
    rows = np.asarray(rows, dtype=np.int64)
    col0 = np.asarray(col0, dtype=np.int64)
    cols = (col0[:, None] + np.arange(width)[None, :]).reshape(-1)
    return dw_at(dy_bits, x_bits, np.repeat(rows, width), cols).reshape(rows.shape[0], width)


def apply_update(opt: str, g, w_bits, m, v, hp, t: int, seed: int, e,
                 state: str = "fp32", m_scales=None, v_scales=None) -> Dict[str, Optional[np.ndarray]]:
    """Steps 2-5 on binary32 gradients ``g`` at flat weight indices ``e`` (same shape as g).

    For ``state == "int8"`` the last axis of every array is a whole number of
    64-element blocks and ``m_scales``/``v_scales`` hold one scale per block.
    For ``state == "bf16"`` m and v are bfloat16 bit patterns.
    Returns W (bf16 bits), w_f32 (the binary32 weight before rounding), m, v and,
    for INT8 states, m_scales and v_scales; for INT8 and BF16 states also m_f32
    and v_f32, the binary32 moments before quantisation or rounding.
    """
    use_m, use_v = optim.USES[opt]
    if state == "int8":
        m32 = int8_block.dequantize(m, m_scales) if use_m else None
        v32 = int8_block.dequantize(v, v_scales) if use_v else None
    elif state == "bf16":
        m32 = bf16.to_f32(m) if use_m else None
        v32 = bf16.to_f32(v) if use_v else None
    else:
        m32 = np.asarray(m, dtype=np.float32) if use_m else None
        v32 = np.asarray(v, dtype=np.float32) if use_v else None
    w64 = bf16.to_f64(w_bits)
    w1, m1, v1 = optim.update(opt, np.asarray(g, dtype=np.float32).astype(np.float64), w64,
                              None if m32 is None else m32.astype(np.float64),
                              None if v32 is None else v32.astype(np.float64), hp, t)
    w1_32 = w1.astype(np.float32)
    e = np.asarray(e, dtype=np.uint64)
    r = philox.sr_bits(seed, t, e.reshape(-1)).reshape(e.shape)
    out: Dict[str, Optional[np.ndarray]] = {
        "W": bf16.stochastic_round(w1_32, r), "w_f32": w1_32,
        "m": None, "v": None, "m_scales": None, "v_scales": None,
    }
    m1_32 = None if m1 is None else m1.astype(np.float32)
    v1_32 = None if v1 is None else v1.astype(np.float32)
    if state == "int8":
        if m1_32 is not None:
            out["m"], out["m_scales"] = int8_block.quantize(m1_32)
        if v1_32 is not None:
            out["v"], out["v_scales"] = int8_block.quantize(v1_32)
        out["m_f32"], out["v_f32"] = m1_32, v1_32
    elif state == "bf16":
        flat = e.reshape(-1)
        if m1_32 is not None:
            out["m"] = bf16.stochastic_round(m1_32, philox.sr_bits(seed, t, flat, philox.STREAM_M).reshape(e.shape))
        if v1_32 is not None:
            out["v"] = bf16.stochastic_round(v1_32, philox.sr_bits(seed, t, flat, philox.STREAM_V).reshape(e.shape))
        out["m_f32"], out["v_f32"] = m1_32, v1_32
    else:
        out["m"], out["v"] = m1_32, v1_32
    return out


def fused_step(opt: str, dy_bits, x_bits, w_bits, m, v, hp, t: int, seed: int,
               state: str = "fp32", m_scales=None, v_scales=None) -> Dict[str, Optional[np.ndarray]]:
    """The whole step on a full layer; arrays keep their [d_out, d_in] shapes."""
    w_bits = np.asarray(w_bits, dtype=np.uint16)
    d_out, d_in = w_bits.shape
    g = dw(dy_bits, x_bits)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    out = apply_update(opt, g, w_bits, m, v, hp, t, seed, e, state, m_scales, v_scales)
    out["g"] = g
    return out


def fused_step_at(opt: str, dy_bits, x_bits, w_bits, m, v, hp, t: int, seed: int,
                  rows: Sequence[int], cols: Sequence[int], state: str = "fp32") -> Dict[str, Optional[np.ndarray]]:
    """The step at sampled positions of a large layer (binary32 or BF16 states)."""
    assert state in ("fp32", "bf16")
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    d_in = np.asarray(w_bits).shape[1]
    g = dw_at(dy_bits, x_bits, rows, cols)
    pick = lambda a: None if a is None else np.asarray(a)[rows, cols]
    e = (rows * d_in + cols).astype(np.uint64)
    out = apply_update(opt, g, pick(w_bits), pick(m), pick(v), hp, t, seed, e, state)
    out["g"] = g
    return out


def fused_step_blocks(opt: str, dy_bits, x_bits, w_bits, m, v, hp, t: int, seed: int,
                      rows: Sequence[int], col0: Sequence[int], m_scales=None, v_scales=None,
                      ) -> Dict[str, Optional[np.ndarray]]:
    """The step on sampled 64-element blocks of a large layer with INT8 states.

    ``m_scales``/``v_scales`` are the full [d_out, d_in/64] scale arrays.
    """
    rows = np.asarray(rows, dtype=np.int64)
    col0 = np.asarray(col0, dtype=np.int64)
    d_in = np.asarray(w_bits).shape[1]
    cols = col0[:, None] + np.arange(64)[None, :]
    g = dw_blocks(dy_bits, x_bits, rows, col0)
    pick = lambda a: None if a is None else np.asarray(a)[rows[:, None], cols]
    pick_s = lambda s: None if s is None else np.asarray(s)[rows, col0 // 64][:, None]
    e = (rows[:, None] * d_in + cols).astype(np.uint64)
    out = apply_update(opt, g, pick(w_bits), pick(m), pick(v), hp, t, seed, e, "int8",
                       pick_s(m_scales), pick_s(v_scales))
    out["g"] = g
    return out
