"""FP8 (E4M3) operands for the weight gradient.  TEST INFRASTRUCTURE ONLY (see the package docstring).

FORGE summary, §4 Experimental results, "Composability": FORGE composes with FP8 quantisation
and absorbs the dequantisation cost.  Reading (stated in the design notes): dY and X arrive as
E4M3 codes with one binary32 scale per tensor (value = scale * decode(code)); the dequantisation
is applied once to the FP32 gradient tile, before the optimizer:

  g = binary32( binary32( sum_t dY8[t, o] X8[t, i] ) * s ),   s = binary32(s_dY * s_X),

the sum exact in float64 (E4M3 x E4M3 products have at most 8 significant bits), rounded once to
binary32.  Everything after g is the fused step of ``step.apply_update``.

Per-channel scales (one per column of dY, i.e. per output channel o, and one per column of X, per
input channel i) factor out of the sum over tokens the same way:

  g[o, i] = binary32( binary32( sum_t dY8[t, o] X8[t, i] ) * binary32(s_dY[o] * s_X[i]) ),

of which the per-tensor case is the special case of constant scale vectors.

E4M3 (OCP 8-bit floating point, "E4M3" format): 1 sign bit, 4 exponent bits with bias 7, 3
mantissa bits; exponent field 0 encodes subnormals mantissa/8 * 2^-6; S.1111.111 is NaN; there are
no infinities, and the largest finite magnitude is 1.75 * 2^8 = 448.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from . import step


def decode_e4m3(codes) -> np.ndarray:
    """E4M3 codes (uint8) -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    out = sign * np.where(e == 0, sub, normal)
    out[(c & 0x7F) == 0x7F] = np.nan
    return out


def _scale_product(s_dy, s_x, rows=None, cols=None) -> np.ndarray:
    """binary32 s_dY * s_X: a scalar (per-tensor) or per (row, col) for channel scale vectors."""
    a = np.asarray(s_dy, dtype=np.float32)
    b = np.asarray(s_x, dtype=np.float32)
    if a.ndim == 0 and b.ndim == 0:
        return np.float32(a * b)
    if rows is not None:  # at listed (row, col) positions
        return ((a[rows] if a.ndim else a) * (b[cols] if b.ndim else b)).astype(np.float32)
    return (np.atleast_1d(a)[:, None] * np.atleast_1d(b)[None, :]).astype(np.float32)


def dw_fp8(dy_codes, x_codes, s_dy, s_x) -> np.ndarray:
    """The dequantised weight gradient, binary32 [d_out, d_in]; scales per tensor (floats) or per
    channel (s_dy [d_out], s_x [d_in])."""
    acc = (decode_e4m3(dy_codes).T @ decode_e4m3(x_codes)).astype(np.float32)
    s = _scale_product(s_dy, s_x)
    return (acc.astype(np.float64) * np.asarray(s, np.float64)).astype(np.float32)


def fused_step_fp8(opt: str, dy_codes, x_codes, s_dy, s_x, w_bits, m, v, hp, t: int, seed: int,
                   state: str = "fp32", m_scales=None, v_scales=None) -> Dict[str, Optional[np.ndarray]]:
    """The fused step with FP8 operands on a full layer (arrays keep their [d_out, d_in] shapes)."""
    w_bits = np.asarray(w_bits, dtype=np.uint16)
    d_out, d_in = w_bits.shape
    g = dw_fp8(dy_codes, x_codes, s_dy, s_x)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    out = step.apply_update(opt, g, w_bits, m, v, hp, t, seed, e, state, m_scales, v_scales)
    out["g"] = g
    return out


def dw_fp8_at(dy_codes, x_codes, s_dy, s_x, rows, cols) -> np.ndarray:
    """dW at listed (row, col) positions, one T-term dot product each."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    a = decode_e4m3(np.asarray(dy_codes)[:, rows])
    b = decode_e4m3(np.asarray(x_codes)[:, cols])
    acc = np.einsum("tn,tn->n", a, b).astype(np.float32)
    s = _scale_product(s_dy, s_x, rows, cols)
    return (acc.astype(np.float64) * np.asarray(s, np.float64)).astype(np.float32)
