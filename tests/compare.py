"""Parity criteria between the CUDA path and the oracle.

* bfloat16 weights: every element within one bfloat16 ULP of the oracle's, and at
  least 99.9 % bit-identical (both sides draw the same Philox bits, so they differ
  only where the binary32 weight before rounding differs by a few ULP across a
  rounding boundary).  Where the new weight nearly cancels (W' = W - dW with
  |W'| << |W|), a binary32 computation of W' carries an error of a few binary32
  ULP of |W| itself, which can exceed a bfloat16 ULP of the tiny result; there the
  bound is the arithmetic's own, 8 binary32 roundings of |W_old|: the tolerance is
  ulp_bf16(ref) + 2^-21 |W_old|.  For every element that does not cancel this term
  is far below one bfloat16 ULP, so the criterion is the 1-ULP one.  At long token
  runs the gradient's own allowed deviation (below) also moves W'; the oracle then
  measures that movement itself (gradient_sensitivity) and it is added.
* binary32 moments: |gpu - ref| <= rtol * max(|ref|, rms(ref)).  A pure relative
  bound is unreachable where dY^T X nearly cancels, because the summation order
  over tokens differs (the summary's exactness statement allows exactly that
  difference); the rms floor bounds the error by the tensor's own scale.
  rtol(T) = max(1e-5, 0.75 (T/16) 2^-23), from the tensor core's accumulation as
  measured (tests/tensor_core_sum.py reproduces the GPU's dW bit for bit): every
  16-token MMA truncates its terms and its sum toward zero, so the deviation from
  the exact sum grows with T/16; its largest value relative to max(|ref|, rms(ref))
  is 0.47-0.6 (T/16) 2^-23 on the workloads (up to 1.4e-5 for the Llama layers at
  T = 4096, against the specification's 1e-5), which tests/test_tensor_core_sum.py
  and tests/test_gpu_tensor_core_sum.py check against this bound.  For T <= 1789
  it is the specification's 1e-5.  v, which squares g, gets twice the bound.
* INT8 codes within +-1; their scales within the moment tolerance.
* bfloat16 moments (BF16 states) are rounded stochastically like the weight: the weight's
  criterion applies, with the moment before the step in place of W_old and the moment's own
  gradient sensitivity.  The bit-identical fraction required of either is 99.9 % less the
  expected share of rounding flips that sensitivity causes (assert_weights).
"""
import numpy as np

from oracle import bf16

W_IDENTICAL_FRACTION = 0.999
MOMENT_RTOL = 1e-5
# largest deviation of the tensor core's sum from the exact one, relative to max(|ref|, rms(ref)),
# in units of (T/16) 2^-23 (one binary32 ULP per 16-token MMA), with a margin
TC_DEVIATION = 0.75


def moment_rtol(T: int, squared: bool = False) -> float:
    """Tolerance for a binary32 quantity linear in g (squared: quadratic in g) at T tokens."""
    r = max(MOMENT_RTOL, TC_DEVIATION * (T / 16) * 2.0 ** -23)
    return 2 * r if squared else r


def assert_weights(gpu_bits, ref_bits, what="W", w_old_bits=None, extra_tol=None):
    """extra_tol: per-element absolute allowance for the movement of the binary32 weight that the
    gradient's allowed summation deviation causes (gradient_sensitivity).

    Stochastic rounding with the same 16 random bits sends two binary32 values that are d apart to
    different bfloat16 neighbours with probability d / ulp.  So where the allowed movement is a
    sizeable part of an ULP (BF16 moments at long token runs, whose value moves in proportion to
    g), the bit-identical fraction is lowered by its expected cost, mean(min(1, extra_tol / ulp)),
    below the 99.9 %."""
    g = np.asarray(gpu_bits, np.uint16).ravel()
    r = np.asarray(ref_bits, np.uint16).ravel()
    assert g.shape == r.shape
    same = g == r
    frac = same.mean()
    gv, rv = bf16.to_f64(g), bf16.to_f64(r)
    ulp = bf16.ulp(r)
    tol = np.where(r & 0x7FFF == 0, bf16.to_f64(np.uint16(1)), ulp)  # ULP at zero: the smallest subnormal
    if w_old_bits is not None:
        wo = bf16.to_f64(np.asarray(w_old_bits, np.uint16).ravel())
        tol = tol + 2.0 ** -21 * np.abs(wo)
    if extra_tol is not None:
        tol = tol + np.asarray(extra_tol, np.float64).ravel()
    bad = ~same & ~(np.abs(gv - rv) <= tol)
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond 1 ULP, e.g. idx {np.flatnonzero(bad)[:5]} " \
                          f"gpu {gv[bad][:5]} ref {rv[bad][:5]}"
    need = W_IDENTICAL_FRACTION
    if extra_tol is not None and g.size:
        need -= float(np.mean(np.minimum(1.0, np.asarray(extra_tol, np.float64).ravel() / ulp)))
    assert frac >= need, f"{what}: only {frac:.6f} bit-identical (at least {need:.6f} required)"
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


def gradient_sensitivity(opt, g, w_bits, m, v, hp, t, seed, e, rtol, state="fp32", m_scales=None, v_scales=None,
                         what="w_f32"):
    """Per element, how far the oracle's binary32 output `what` (the weight, or m_f32 / v_f32 for
    rounded states) moves when its gradient moves by the summation deviation the summary allows,
    rtol * max(|g|, rms(g)), in either direction.  Used as an extra tolerance: the GPU must agree,
    within one bfloat16 ULP, with the oracle evaluated at some gradient inside that band.  (For
    Lion this includes a sign flip of c.)"""
    from oracle import step as ostep
    g64 = np.asarray(g, np.float64)
    band = rtol * np.maximum(np.abs(g64), np.sqrt(np.mean(g64 * g64)))
    base = ostep.apply_update(opt, g, w_bits, m, v, hp, t, seed, e, state, m_scales, v_scales)[what]
    out = np.zeros(g64.shape)
    for sign in (-1.0, 1.0):
        moved = ostep.apply_update(opt, (g64 + sign * band).astype(np.float32), w_bits, m, v, hp, t, seed, e,
                                   state, m_scales, v_scales)[what]
        out = np.maximum(out, np.abs(moved.astype(np.float64) - base.astype(np.float64)))
    return out


DX_IDENTICAL_FRACTION = 0.99


def assert_bf16_sum(gpu_bits, ref_f32, K, what="dX"):
    """A K-term sum accumulated in FP32 and rounded once, to nearest even, to bfloat16.

    ref_f32 is the exact sum rounded to binary32; its round-to-nearest-even bfloat16 is the
    expected value.  The GPU's FP32 sum may differ from it by the accumulator's allowed deviation
    rt * max(|ref|, rms(ref)), rt = moment_rtol(K) (the same reading as for dW), which moves the
    bfloat16 result across a rounding boundary where the sum lies within that distance of one:
    tolerance = one bfloat16 ULP + that deviation, and at least 99 % of elements bit-identical."""
    g = np.asarray(gpu_bits, np.uint16).ravel()
    r32 = np.asarray(ref_f32, np.float32).ravel()
    r = bf16.round_nearest_even(r32)
    same = g == r
    frac = float(same.mean()) if same.size else 1.0
    rv = r32.astype(np.float64)
    scale = np.maximum(np.abs(rv), np.sqrt(np.mean(rv * rv)) if rv.size else 0.0)
    ulp = np.where(r & 0x7FFF == 0, bf16.to_f64(np.uint16(1)), bf16.ulp(r))
    tol = ulp + moment_rtol(K) * scale
    bad = ~same & ~(np.abs(bf16.to_f64(g) - rv) <= tol)
    assert not bad.any(), f"{what}: {bad.sum()} of {g.size} beyond tolerance, e.g. idx {np.flatnonzero(bad)[:5]} " \
                          f"gpu {bf16.to_f64(g)[bad][:5]} ref {rv[bad][:5]}"
    assert frac >= DX_IDENTICAL_FRACTION, f"{what}: only {frac:.6f} bit-identical"
    return frac


def assert_codes(gpu, ref, what="codes"):
    d = np.abs(np.asarray(gpu, np.int64) - np.asarray(ref, np.int64))
    assert d.max(initial=0) <= 1, f"{what}: code difference {d.max()}"
    return float((d == 0).mean()) if d.size else 1.0
