"""Pins for the oracle's FP8 (E4M3) operands (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8, step
from workloads import default_hparams, fp8_e4m3


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_decode_all_codes(decode):
    """Every one of the 256 codes against PyTorch's float8_e4m3fn (NaN codes: both NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    np.testing.assert_array_equal(decode(codes), _torch_decode(codes))


def pin_decode_landmarks(decode):
    """Values the format's definition fixes: 1, the largest finite, the smallest normal and
    subnormal, negative zero, and NaN."""
    got = decode(np.array([0x38, 0x7E, 0x08, 0x01, 0x80, 0xFE, 0x7F], np.uint8))
    np.testing.assert_array_equal(got[:6], [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, 0.0, -448.0])
    assert np.signbit(got[4]) and np.isnan(got[6])


DECODE_PINS = [pin_decode_all_codes, pin_decode_landmarks]


@pytest.mark.parametrize("pin", DECODE_PINS, ids=lambda p: p.__name__)
def test_decode_pins(pin):
    pin(fp8.decode_e4m3)


@pytest.mark.parametrize("kind", ["bias_8", "no_subnormals", "four_mantissa_steps"])
def test_decode_pins_catch_planted_mistakes(kind):
    def decode(codes):
        c = np.asarray(codes, np.uint8).astype(np.int64)
        s = np.where(c & 0x80, -1.0, 1.0)
        e, m = (c >> 3) & 0xF, c & 7
        bias, frac = (8, 8.0) if kind == "bias_8" else (7, 4.0 if kind == "four_mantissa_steps" else 8.0)
        v = np.ldexp(1 + m / frac, e - bias)
        if kind != "no_subnormals":
            v = np.where(e == 0, np.ldexp(m / frac, 1 - bias), v)
        out = s * v
        out[(c & 0x7F) == 0x7F] = np.nan
        return out
    with pytest.raises(AssertionError):
        for pin in DECODE_PINS:
            pin(decode)


def test_dw_fp8_brute_force():
    """Exact rational sums of decoded products, rounded once to binary32, times the binary32 scale product."""
    rng = np.random.default_rng(1)
    dy = rng.integers(0, 256, size=(7, 3)).astype(np.uint8)
    x = rng.integers(0, 256, size=(7, 5)).astype(np.uint8)
    dy[(dy & 0x7F) == 0x7F] = 0x38  # no NaN codes
    x[(x & 0x7F) == 0x7F] = 0x30
    s_dy, s_x = 3.0e-5, 0.7
    got = fp8.dw_fp8(dy, x, s_dy, s_x)
    a, b = _torch_decode(dy), _torch_decode(x)
    s = np.float32(np.float32(s_dy) * np.float32(s_x))
    for o in range(3):
        for i in range(5):
            exact = sum(Fraction(float(a[t, o])) * Fraction(float(b[t, i])) for t in range(7))
            want = np.float32(float(np.float32(float(exact))) * float(s))
            assert got[o, i] == want, (o, i)


def test_dw_fp8_power_of_two_scales_are_exact_shifts():
    rng = np.random.default_rng(2)
    dy = rng.integers(0, 0x70, size=(64, 8)).astype(np.uint8)
    x = rng.integers(0, 0x70, size=(64, 16)).astype(np.uint8)
    base = fp8.dw_fp8(dy, x, 1.0, 1.0)
    np.testing.assert_array_equal(fp8.dw_fp8(dy, x, 2.0 ** -7, 2.0 ** 3), base * np.float32(2.0 ** -4))
    rows, cols = np.array([0, 7, 3]), np.array([15, 0, 8])
    np.testing.assert_array_equal(fp8.dw_fp8_at(dy, x, 2.0 ** -7, 2.0 ** 3, rows, cols),
                                  (base * np.float32(2.0 ** -4))[rows, cols])


def test_quantised_inputs_round_trip_within_half_a_step():
    """The input generator's codes decode to within half an E4M3 step of t / scale."""
    t = torch.randn(4096, generator=torch.Generator().manual_seed(3)) * 1e-3
    codes, scale = fp8_e4m3(t)
    back = fp8.decode_e4m3(codes.numpy()) * scale
    ref = t.double().numpy()
    step_size = np.maximum(np.abs(ref), 2.0 ** -6 * scale) * 2.0 ** -3
    assert np.all(np.abs(back - ref) <= 0.5 * step_size + 1e-30)
    assert np.abs(fp8.decode_e4m3(codes.numpy())).max() == 448.0


def test_fused_step_fp8_is_the_update_on_the_dequantised_gradient():
    rng = np.random.default_rng(4)
    dy = rng.integers(0, 0x70, size=(32, 16)).astype(np.uint8)
    x = rng.integers(0, 0x70, size=(32, 24)).astype(np.uint8)
    w = rng.integers(0x3C00, 0x3D00, size=(16, 24)).astype(np.uint16)
    m = np.zeros((16, 24), np.float32)
    v = np.zeros((16, 24), np.float32)
    hp = default_hparams("adamw", lr=1e-3)
    out = fp8.fused_step_fp8("adamw", dy, x, 1e-2, 2e-3, w, m, v, hp, 1, 5)
    e = np.arange(16 * 24, dtype=np.uint64).reshape(16, 24)
    ref = step.apply_update("adamw", fp8.dw_fp8(dy, x, 1e-2, 2e-3), w, m, v, hp, 1, 5, e)
    np.testing.assert_array_equal(out["W"], ref["W"])
    np.testing.assert_array_equal(out["m"], ref["m"])


def test_channel_scales_reduce_to_the_tensor_scale():
    rng = np.random.default_rng(5)
    dy = rng.integers(0, 0x70, size=(48, 16)).astype(np.uint8)
    x = rng.integers(0, 0x70, size=(48, 24)).astype(np.uint8)
    got = fp8.dw_fp8(dy, x, np.full(16, 3e-4, np.float32), np.full(24, 0.7, np.float32))
    np.testing.assert_array_equal(got, fp8.dw_fp8(dy, x, 3e-4, 0.7))


def test_channel_scales_brute_force_and_orientation():
    """s_dy scales rows of dW (output channels), s_x its columns; exact rational sums, one binary32
    rounding, then the binary32 product of the two channel scales."""
    rng = np.random.default_rng(6)
    dy = rng.integers(0, 0x70, size=(9, 5)).astype(np.uint8)
    x = rng.integers(0, 0x70, size=(9, 5)).astype(np.uint8)  # square, so a swap would not show in shapes
    s_dy = (rng.random(5) * 1e-3 + 1e-4).astype(np.float32)
    s_x = (rng.random(5) + 0.5).astype(np.float32)
    got = fp8.dw_fp8(dy, x, s_dy, s_x)
    a, b = _torch_decode(dy), _torch_decode(x)
    for o in range(5):
        for i in range(5):
            exact = sum(Fraction(float(a[t, o])) * Fraction(float(b[t, i])) for t in range(9))
            s = np.float32(s_dy[o] * s_x[i])
            assert got[o, i] == np.float32(float(np.float32(float(exact))) * float(s)), (o, i)
    rows, cols = np.array([4, 0, 2]), np.array([1, 3, 4])
    np.testing.assert_array_equal(fp8.dw_fp8_at(dy, x, s_dy, s_x, rows, cols), got[rows, cols])


def test_channel_quantised_inputs_round_trip():
    from workloads import fp8_e4m3_channels
    t = torch.randn(256, 40, generator=torch.Generator().manual_seed(7)) * torch.logspace(-4, 0, 40)[None, :]
    codes, scale = fp8_e4m3_channels(t)
    back = fp8.decode_e4m3(codes.numpy()) * scale.numpy()[None, :]
    assert np.abs(fp8.decode_e4m3(codes.numpy())).max(axis=0).tolist() == [448.0] * 40
    rel = np.abs(back - t.double().numpy()) / np.maximum(np.abs(t.double().numpy()), 2.0 ** -6 * scale.numpy()[None, :])
    assert rel.max() <= 2.0 ** -4 + 1e-12
