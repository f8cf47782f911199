"""Pins for the oracle's bfloat16 encoding and stochastic rounding (CPU only)."""
import numpy as np
import torch

from oracle import bf16


def test_bits_roundtrip_against_torch_bfloat16():
    x = torch.randn(10_000, generator=torch.Generator().manual_seed(0)) * 3
    b = x.to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16.to_f32(bits), b.float().numpy())


def test_round_nearest_even_matches_torch_cast():
    g = torch.Generator().manual_seed(1)
    x = torch.cat([torch.randn(100_000, generator=g) * 10.0 ** torch.randint(-30, 30, (100_000,), generator=g),
                   torch.tensor([0.0, -0.0, float("inf"), float("-inf"), 3.3895314e38, 1e-40])])
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16.round_nearest_even(x.numpy()), ref)


def test_stochastic_rounding_expectation_is_exact():
    """Over all 2^16 random values, the mean of SR(x) is x exactly (exact rational check)."""
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(200).astype(np.float32) * 0.02,
                         np.array([1.0 + 2.0 ** -20, -3.0000002, 1e-30], np.float32)])
    r = np.arange(65536, dtype=np.uint32)
    for x in xs:
        out = bf16.to_f64(bf16.stochastic_round(np.full(65536, x, np.float32), r))
        # sum of 2^16 doubles each with <= 8 significant bits: exact in float64
        assert out.sum() / 65536.0 == float(x), x


def test_stochastic_rounding_rounds_to_neighbours_with_right_probability():
    x = np.float32(1.0 + 2.0 ** -9)  # 1/4 of the way from 1.0 to the next bf16 (1 + 2^-7)
    r = np.arange(65536, dtype=np.uint32)
    out = bf16.to_f64(bf16.stochastic_round(np.full(65536, x, np.float32), r))
    vals, counts = np.unique(out, return_counts=True)
    assert vals.tolist() == [1.0, 1.0 + 2.0 ** -7]
    assert counts.tolist() == [49152, 16384]


def test_exact_values_and_specials_are_unchanged():
    r = np.array([0, 1, 0x7FFF, 0xFFFF], np.uint32)
    for v in [0.0, -0.0, 1.0, -2.5, 0.015625, float("inf"), float("-inf")]:
        out = bf16.stochastic_round(np.full(4, v, np.float32), r)
        assert np.all(bf16.to_f32(out) == np.float32(v))
        assert np.all(np.signbit(bf16.to_f32(out)) == np.signbit(np.float32(v)))
    nan = bf16.stochastic_round(np.array([np.nan, -np.nan], np.float32), np.array([5, 0xFFFF], np.uint32))
    assert nan.tolist() == [0x7FC0, 0x7FC0]


def test_dead_zone_control():
    """A sub-ULP update vanishes under round-to-nearest but accumulates under SR."""
    w0 = np.float32(0.02)
    ulp = bf16.ulp(bf16.round_nearest_even(w0))[()]
    delta = ulp * 1e-2
    w_rne = bf16.round_nearest_even(w0)
    w_sr = bf16.round_nearest_even(w0)
    rng = np.random.default_rng(3)
    for _ in range(1000):
        w_rne = bf16.round_nearest_even(bf16.to_f32(w_rne) + np.float32(delta))
        w_sr = bf16.stochastic_round(bf16.to_f32(w_sr) + np.float32(delta),
                                     rng.integers(0, 65536, size=w_sr.shape, dtype=np.uint32))
    assert bf16.to_f64(w_rne)[()] == bf16.to_f64(bf16.round_nearest_even(w0))[()]
    drift = bf16.to_f64(w_sr)[()] - float(w0)
    assert 3 * ulp <= drift <= 20 * ulp  # expectation 10 ULP
