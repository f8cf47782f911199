"""Parity criteria between the CUDA path and the oracle.

* bfloat16 weights: every element within one bfloat16 ULP of the oracle's, and at
  least 99.9 % bit-identical (both sides draw the same Philox bits, so they differ
  only where the binary32 weight before rounding differs by a few ULP across a
  rounding boundary).  Where the new weight nearly cancels (W' = W - dW with
  |W'| << |W|), a binary32 computation of W' carries an error of a few binary32
  ULP of |W| itself, which can exceed a bfloat16 ULP of the tiny result; there the
  bound is the arithmetic's own, 8 binary32 roundings of |W_old|: the tolerance is
  ulp_bf16(ref) + 2^-21 |W_old|.  For every element that does not cancel this term
  is far below one bfloat16 ULP, so the criterion is the 1-ULP one.
* binary32 moments: |gpu - ref| <= 1e-5 * max(|ref|, rms(ref)).  A pure relative
  bound is unreachable where dY^T X nearly cancels, because the summation order
  over tokens differs (the summary's exactness statement allows exactly that
  difference); the rms floor bounds the error by the tensor's own scale.
* INT8 codes within +-1; their scales within the moment tolerance.
"""
import numpy as np

from oracle import bf16

W_IDENTICAL_FRACTION = 0.999
MOMENT_RTOL = 1e-5


def assert_weights(gpu_bits, ref_bits, what="W", w_old_bits=None):
    g = np.asarray(gpu_bits, np.uint16).ravel()
    r = np.asarray(ref_bits, np.uint16).ravel()
    assert g.shape == r.shape
    same = g == r
    frac = same.mean()
    gv, rv = bf16.to_f64(g), bf16.to_f64(r)
    ulp = bf16.ulp(r)
    tol = np.where(r & 0x7FFF == 0, bf16.to_f64(np.uint16(1)), ulp)  # ULP at zero: the smallest subnormal
    if w_old_bits is not None:
        tol = tol + 2.0 ** -21 * np.abs(bf16.to_f64(np.asarray(w_old_bits, np.uint16).ravel()))
    bad = ~same & ~(np.abs(gv - rv) <= tol)
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond 1 ULP, e.g. idx {np.flatnonzero(bad)[:5]} " \
                          f"gpu {gv[bad][:5]} ref {rv[bad][:5]}"
    assert frac >= W_IDENTICAL_FRACTION, f"{what}: only {frac:.6f} bit-identical"
    return frac


def assert_moments(gpu, ref, what="m", rtol=MOMENT_RTOL):
    g = np.asarray(gpu, np.float64).ravel()
    r = np.asarray(ref, np.float64).ravel()
    scale = np.maximum(np.abs(r), np.sqrt(np.mean(r * r)) if r.size else 0.0)
    err = np.abs(g - r)
    bad = err > rtol * scale
    assert not bad.any(), f"{what}: {bad.sum()} of {r.size} beyond tolerance, max err/scale " \
                          f"{(err / np.where(scale > 0, scale, 1)).max():.3e}, e.g. gpu {g[bad][:4]} ref {r[bad][:4]}"
    return float((err / np.where(scale > 0, scale, 1)).max()) if r.size else 0.0


def assert_codes(gpu, ref, what="codes"):
    d = np.abs(np.asarray(gpu, np.int64) - np.asarray(ref, np.int64))
    assert d.max(initial=0) <= 1, f"{what}: code difference {d.max()}"
    return float((d == 0).mean()) if d.size else 1.0
