"""Pins for the oracle's input gradient dX = dY W and the layer backward (CPU only).

Each pin takes the dx function under test, so planted mistakes (a transposed W, a
truncating or missing bfloat16 rounding, dY^T in place of dY) can be run through the
same pins and must fail one of them.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import backward, bf16, step
from tests.helpers import bits, f32
from workloads import default_hparams, normal_bf16


def _bf16_bits_torch(x_f32):
    """binary32 -> bfloat16 bits through PyTorch's own conversion (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def pin_brute_force(dx):
    """Exact rational sums in a triple loop, one rounding to binary32, then PyTorch's RNE."""
    dy = bits(normal_bf16((5, 7), 1e-2, seed=11))
    w = bits(normal_bf16((7, 3), 1.0, seed=12))
    dyf, wf = bf16.to_f32(dy), bf16.to_f32(w)
    ref = np.empty((5, 3), np.float32)
    for t in range(5):
        for i in range(3):
            s = Fraction(0)
            for o in range(7):
                s += Fraction(float(dyf[t, o])) * Fraction(float(wf[o, i]))
            ref[t, i] = np.float32(float(s))
    got = dx(dy, w)
    assert got.shape == (5, 3)
    np.testing.assert_array_equal(got, _bf16_bits_torch(ref))


def pin_identity_and_permutation(dx):
    """W = I gives dY back bit for bit; a permutation matrix moves columns the documented way."""
    dy = bits(normal_bf16((6, 8), 0.5, seed=13))
    eye = bf16.round_nearest_even(np.eye(8, dtype=np.float32))
    np.testing.assert_array_equal(dx(dy, eye), dy)
    perm = np.array([3, 0, 6, 1, 7, 2, 5, 4])  # W[o, perm[o]] = 1, so dX[:, perm[o]] = dY[:, o]
    p = np.zeros((8, 8), np.float32)
    p[np.arange(8), perm] = 1.0
    out = dx(dy, bf16.round_nearest_even(p))
    np.testing.assert_array_equal(out[:, perm], dy)


def pin_ties_round_to_even(dx):
    """1 + 2^-8 and 1 + 3*2^-8 lie halfway between bfloat16 neighbours: they round to the even one."""
    dy = bf16.round_nearest_even(np.array([[1.0, 2.0 ** -8], [1.0, 3 * 2.0 ** -8], [-1.0, -(2.0 ** -8)]], np.float32))
    w = bf16.round_nearest_even(np.array([[1.0], [1.0]], np.float32))
    got = bf16.to_f64(dx(dy, w)).ravel()
    np.testing.assert_array_equal(got, [1.0, 1.0 + 2.0 ** -6, -1.0])


def pin_against_torch(dx):
    """Float64 matmul in PyTorch, cast to binary32, then PyTorch's bfloat16 conversion."""
    dy = bits(normal_bf16((96, 40), 1e-3, seed=14))
    w = bits(normal_bf16((40, 24), 2e-2, seed=15))
    ref = (torch.from_numpy(bf16.to_f64(dy)) @ torch.from_numpy(bf16.to_f64(w))).float().numpy()
    np.testing.assert_array_equal(dx(dy, w), _bf16_bits_torch(ref))


PINS = [pin_brute_force, pin_identity_and_permutation, pin_ties_round_to_even, pin_against_torch]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_dx_pins(pin):
    pin(backward.dx)


def _mutant(kind):
    def dx(dy_bits, w_bits):
        dy, w = bf16.to_f64(dy_bits), bf16.to_f64(w_bits)
        if kind == "transposed_w":
            r = dy @ w.T if w.shape[0] == w.shape[1] else dy @ w
            return bf16.round_nearest_even(r.astype(np.float32))
        if kind == "truncated":
            return (bf16.f32_bits((dy @ w).astype(np.float32)) >> 16).astype(np.uint16)
        if kind == "round_half_up":
            u = bf16.f32_bits((dy @ w).astype(np.float32)).astype(np.uint64)
            return ((u + 0x8000) >> 16).astype(np.uint16)
        if kind == "bf16_accumulate":
            acc = np.zeros((dy.shape[0], w.shape[1]), np.float32)
            for o in range(dy.shape[1]):
                acc = bf16.to_f32(bf16.round_nearest_even(acc + np.outer(dy[:, o], w[o]).astype(np.float32)))
            return bf16.round_nearest_even(acc)
        raise ValueError(kind)
    return dx


@pytest.mark.parametrize("kind", ["transposed_w", "truncated", "round_half_up", "bf16_accumulate"])
def test_dx_pins_catch_planted_mistakes(kind):
    failed = 0
    for pin in PINS:
        try:
            pin(_mutant(kind))
        except AssertionError:
            failed += 1
    assert failed > 0, f"no pin caught {kind}"


def test_dx_at_samples_the_full_product():
    dy = bits(normal_bf16((64, 96), 1e-3, seed=16))
    w = bits(normal_bf16((96, 48), 2e-2, seed=17))
    full = backward.dx(dy, w)
    rows = np.array([0, 5, 63, 17, 40])
    cols = np.array([0, 47, 3, 20, 47])
    got = backward.dx_at(dy, w, rows, cols)
    np.testing.assert_array_equal(got["bits"], full[rows, cols])


def test_linear_backward_reads_the_weights_before_the_step():
    """dX comes from W_old (it differs from dY W_new), and the weight step is the fused step's."""
    T, d_out, d_in = 32, 16, 24
    dy = bits(normal_bf16((T, d_out), 1e-2, seed=18))
    x = bits(normal_bf16((T, d_in), 1.0, seed=19))
    w = bits(normal_bf16((d_out, d_in), 2e-2, seed=20))
    m = np.zeros((d_out, d_in), np.float32)
    v = np.zeros((d_out, d_in), np.float32)
    hp = default_hparams("adamw", lr=0.05)
    out = backward.linear_backward("adamw", dy, x, w, m, v, hp, 1, 7)
    np.testing.assert_array_equal(out["dX"], backward.dx(dy, w))
    assert not np.array_equal(out["dX"], backward.dx(dy, out["W"]))
    ref = step.fused_step("adamw", dy, x, w, m, v, hp, 1, 7)
    np.testing.assert_array_equal(out["W"], ref["W"])
    np.testing.assert_array_equal(out["m"], ref["m"])
    np.testing.assert_array_equal(out["v"], ref["v"])
