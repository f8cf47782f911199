"""bfloat16 encoding and the stochastic rounding of the weight write-back.

A bfloat16 is the upper 16 bits of an IEEE-754 binary32 (1 sign, 8 exponent, 7
fraction bits).  Arrays of bfloat16 are carried here as their uint16 bit
patterns so that no library conversion stands between the oracle and the
definition.

Stochastic rounding (FORGE summary, §2 Precision and fidelity, second
low-precision point: weights are written back with stochastic rounding so that
updates smaller than one bfloat16 ULP accumulate without bias instead of
vanishing in the round-to-nearest "dead zone").  The summary gives no bit
recipe; we take the plainest one: add 16 uniform random bits to the binary32
pattern and keep the upper half.  For a finite x between two neighbouring
bfloat16 values lo < x < hi (same sign), this rounds the magnitude up with
probability (|x| - |lo|) / ULP exactly, so E[SR(x)] = x.  NaN maps to the
canonical quiet NaN 0x7FC0, +-Inf stay +-Inf, and values within one ULP of the
largest finite bfloat16 may round to Inf, as round-to-nearest does.

Pinned by: exact expectation over all 2^16 random values, the dead-zone control
with round-to-nearest-even, and bit-pattern special cases (tests/test_oracle_rounding.py).
"""
from __future__ import annotations

import numpy as np


def to_f32(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float32 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def to_f64(bits) -> np.ndarray:
    return to_f32(bits).astype(np.float64)


def f32_bits(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)


def round_nearest_even(x) -> np.ndarray:
    """binary32 -> bfloat16 bits with round-to-nearest-even (the dead-zone control)."""
    u = f32_bits(x).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    r[nan.reshape(r.shape)] = np.uint16(0x7FC0)
    return r


def stochastic_round(x, r16) -> np.ndarray:
    """binary32 values ``x`` -> bfloat16 bits, using 16 random bits ``r16`` per element."""
    x = np.asarray(x, dtype=np.float32)
    u = f32_bits(x).astype(np.uint64)
    exp_all_ones = (u & np.uint64(0x7F800000)) == np.uint64(0x7F800000)
    add = np.where(exp_all_ones, np.uint64(0), np.asarray(r16, dtype=np.uint64) & np.uint64(0xFFFF))
    out = ((u + add) >> np.uint64(16)).astype(np.uint16)
    out[np.isnan(x)] = np.uint16(0x7FC0)
    return out


def ulp(bits) -> np.ndarray:
    """Distance from a finite nonzero bfloat16 to the next one away from zero (float64)."""
    b = np.asarray(bits, dtype=np.uint16)
    nxt = (b.astype(np.uint32) + 1).astype(np.uint16)
    return np.abs(to_f64(nxt) - to_f64(b))
