"""Pins for BF16 optimizer states with stochastic rounding (CPU only).

The update itself is the pinned FP32 one; what BF16 states add is how the new moments are
stored: rounded to binary32, then stochastically to bfloat16 with 16 bits from their own Philox
streams (1 for m, 2 for v; the weight keeps stream 0).  The pins check what that reading fixes:
stream 0 is the pinned weight stream, each stream's bits are uniform, the three tensors round
independently of one another, the rounding is unbiased, exact values stay exact, and the weight
and the binary32 moments are those of the FP32-state update on the decoded moments.  Each pin takes
the update function, so planted mistakes run through the same pins.
"""
import numpy as np
import pytest

from oracle import bf16, philox, step
from workloads import Hparams, default_hparams

N = 1 << 14


def test_stream_zero_is_the_weight_stream():
    e = np.arange(4096, dtype=np.uint64)
    np.testing.assert_array_equal(philox.sr_bits(5, 3, e, philox.STREAM_W), philox.sr_bits(5, 3, e))


@pytest.mark.parametrize("stream", [philox.STREAM_M, philox.STREAM_V])
def test_moment_streams_are_uniform_and_distinct(stream):
    e = np.arange(1 << 16, dtype=np.uint64)
    r = philox.sr_bits(11, 2, e, stream)
    hist = np.bincount((r >> 12).astype(np.int64), minlength=16)  # 16 bins of the top 4 bits
    expected = e.size / 16
    chi2 = float(((hist - expected) ** 2 / expected).sum())
    assert chi2 < 40.0  # 15 degrees of freedom: p < 1e-3 beyond 37.7
    assert (r == philox.sr_bits(11, 2, e, philox.STREAM_W)).mean() < 1e-3


def _same_inputs(opt, w, m, v, g, hp, t=3, seed=9):
    """N elements with identical inputs: only their Philox bits differ."""
    e = np.arange(N, dtype=np.uint64)
    full = lambda x, dt: np.full(N, x, dtype=dt)
    mb = bf16.round_nearest_even(full(m, np.float32))
    vb = bf16.round_nearest_even(full(v, np.float32))
    wb = bf16.round_nearest_even(full(w, np.float32))
    return e, wb, mb, vb, full(g, np.float32), hp, t, seed


def _p_up(x32):
    """Probability that stochastic rounding moves binary32 x away from zero: its low 16 bits / 2^16."""
    return float((bf16.f32_bits(np.asarray(x32, np.float32)).ravel()[0] & 0xFFFF) / 65536.0)


def _up(bits_out, x32):
    return bits_out != (bf16.f32_bits(np.asarray(x32, np.float32)) >> 16).astype(np.uint16)


def _case():
    # values whose binary32 results sit well between bfloat16 neighbours
    hp = Hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    return _same_inputs("adamw", w=0.0123, m=3.1e-4, v=1.9e-7, g=6.1e-4, hp=hp)


def pin_unbiased(apply_update):
    """Mean of the stored moments over elements with equal inputs = the binary32 moment."""
    e, wb, mb, vb, g, hp, t, seed = _case()
    out = apply_update("adamw", g, wb, mb, vb, hp, t, seed, e, "bf16")
    for k in ("m", "v"):
        x = float(out[k + "_f32"][0])
        vals = bf16.to_f64(out[k])
        lo, hi = vals.min(), vals.max()
        assert hi > lo, f"{k}: no element rounded the other way"
        # Bernoulli mean: 5 standard deviations over N draws
        assert abs(vals.mean() - x) <= 5 * (hi - lo) * 0.5 / np.sqrt(N), k


def pin_independent(apply_update):
    """W, m and v round up independently: P(both up) = P(up) P(up) for each pair."""
    e, wb, mb, vb, g, hp, t, seed = _case()
    out = apply_update("adamw", g, wb, mb, vb, hp, t, seed, e, "bf16")
    ups = {"w": _up(out["W"], out["w_f32"]), "m": _up(out["m"], out["m_f32"]), "v": _up(out["v"], out["v_f32"])}
    ps = {"w": _p_up(out["w_f32"]), "m": _p_up(out["m_f32"]), "v": _p_up(out["v_f32"])}
    for k in ps:
        assert 0.05 < ps[k] < 0.95, f"case not informative for {k}"
        assert abs(ups[k].mean() - ps[k]) < 5 * np.sqrt(ps[k] * (1 - ps[k]) / N), k
    for a, b in (("w", "m"), ("w", "v"), ("m", "v")):
        joint = (ups[a] & ups[b]).mean()
        p = ps[a] * ps[b]
        assert abs(joint - p) < 5 * np.sqrt(p * (1 - p) / N) + 1e-3, (a, b, joint, p)


def pin_exact_values_stay(apply_update):
    """beta = 1/2 and g = m = v = 1 give m' = v' = 1 exactly: no random bit may move them."""
    hp = Hparams(lr=1e-3, beta1=0.5, beta2=0.5, eps=1e-8, weight_decay=0.0)
    e, wb, mb, vb, g, hp, t, seed = _same_inputs("adamw", w=0.5, m=1.0, v=1.0, g=1.0, hp=hp)
    out = apply_update("adamw", g, wb, mb, vb, hp, t, seed, e, "bf16")
    assert (bf16.to_f64(out["m"]) == 1.0).all() and (bf16.to_f64(out["v"]) == 1.0).all()


def pin_composes_with_fp32_update(apply_update):
    """Weight and binary32 moments equal the FP32-state update on the decoded moments."""
    rng = np.random.default_rng(3)
    e = np.arange(4096, dtype=np.uint64)
    g = (rng.standard_normal(4096) * 1e-3).astype(np.float32)
    wb = bf16.round_nearest_even((rng.standard_normal(4096) * 2e-2).astype(np.float32))
    mb = bf16.round_nearest_even((rng.standard_normal(4096) * 1e-4).astype(np.float32))
    vb = bf16.round_nearest_even((rng.random(4096) * 1e-6).astype(np.float32))
    for opt in ("adamw", "nadam", "radam", "lion", "rmsprop", "adagrad", "sgd_momentum"):
        hp = default_hparams(opt, lr=1e-3)
        got = apply_update(opt, g, wb, mb, vb, hp, 6, 4, e, "bf16")
        ref = step.apply_update(opt, g, wb, bf16.to_f32(mb), bf16.to_f32(vb), hp, 6, 4, e, "fp32")
        np.testing.assert_array_equal(got["W"], ref["W"])
        for k in ("m", "v"):
            if ref[k] is not None:
                np.testing.assert_array_equal(got[k + "_f32"], ref[k])


PINS = [pin_unbiased, pin_independent, pin_exact_values_stay, pin_composes_with_fp32_update]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_bf16_state_pins(pin):
    pin(step.apply_update)


def _mutant(kind):
    def apply_update(opt, g, w_bits, m, v, hp, t, seed, e, state="fp32", m_scales=None, v_scales=None):
        out = step.apply_update(opt, g, w_bits, m, v, hp, t, seed, e, state, m_scales, v_scales)
        if state != "bf16":
            return out
        flat = np.asarray(e, np.uint64).reshape(-1)
        if kind == "nearest_instead_of_stochastic":
            for k in ("m", "v"):
                if out[k] is not None:
                    out[k] = bf16.round_nearest_even(out[k + "_f32"])
        elif kind == "moments_share_the_weight_stream":
            r = philox.sr_bits(seed, t, flat).reshape(np.shape(e))
            for k in ("m", "v"):
                if out[k] is not None:
                    out[k] = bf16.stochastic_round(out[k + "_f32"], r)
        elif kind == "m_and_v_share_a_stream":
            if out["v"] is not None:
                r = philox.sr_bits(seed, t, flat, philox.STREAM_M).reshape(np.shape(e))
                out["v"] = bf16.stochastic_round(out["v_f32"], r)
        elif kind == "weight_uses_rounded_moments":
            mb = bf16.to_f32(out["m"]) if out["m"] is not None else None
            vb = bf16.to_f32(out["v"]) if out["v"] is not None else None
            # re-derive the weight from the stored (rounded) moments, as a faulty kernel might
            lr = np.float64(np.float32(hp.lr))
            if opt == "adamw" and mb is not None:
                w = bf16.to_f64(w_bits) * (1 - lr * np.float64(np.float32(hp.weight_decay)))
                b1, b2 = np.float64(np.float32(hp.beta1)), np.float64(np.float32(hp.beta2))
                w = w - lr / (1 - b1 ** t) * mb / (np.sqrt(vb / (1 - b2 ** t)) + np.float64(np.float32(hp.eps)))
                out["w_f32"] = w.astype(np.float32)
                out["W"] = bf16.stochastic_round(out["w_f32"], philox.sr_bits(seed, t, flat).reshape(np.shape(e)))
        else:
            raise ValueError(kind)
        return out
    return apply_update


@pytest.mark.parametrize("kind", ["nearest_instead_of_stochastic", "moments_share_the_weight_stream",
                                  "m_and_v_share_a_stream", "weight_uses_rounded_moments"])
def test_bf16_state_pins_catch_planted_mistakes(kind):
    failed = 0
    for pin in PINS:
        try:
            pin(_mutant(kind))
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught {kind}"
