"""Pins for the oracle's weight gradient dW = dY^T X (CPU only)."""
from fractions import Fraction

import numpy as np
import torch

from oracle import bf16, step
from tests.helpers import bits
from workloads import normal_bf16


def _brute_force(dy_bits, x_bits):
    """Triple loop over (o, i, t) with exact rational sums, then one rounding to binary32."""
    dy = bf16.to_f32(dy_bits)
    x = bf16.to_f32(x_bits)
    T, d_out = dy.shape
    d_in = x.shape[1]
    out = np.empty((d_out, d_in), np.float32)
    for o in range(d_out):
        for i in range(d_in):
            s = Fraction(0)
            for t in range(T):
                s += Fraction(float(dy[t, o])) * Fraction(float(x[t, i]))
            out[o, i] = np.float32(float(s))  # Fraction -> nearest double -> binary32
    return out


def test_dw_matches_brute_force_on_non_square_shapes():
    dy = bits(normal_bf16((11, 3), 1e-2, seed=1))
    x = bits(normal_bf16((11, 5), 1.0, seed=2))
    got = step.dw(dy, x)
    ref = _brute_force(dy, x)
    assert got.shape == (3, 5)
    # float64 sum vs exact: at most one binary32 rounding apart (double rounding through float64)
    np.testing.assert_allclose(got, ref, rtol=2 ** -23, atol=0)


def test_dw_integer_inputs_exact():
    rng = np.random.default_rng(0)
    dy = rng.integers(-8, 9, size=(16, 4)).astype(np.float32)
    x = rng.integers(-8, 9, size=(16, 6)).astype(np.float32)
    dyb = bits(torch.from_numpy(dy).to(torch.bfloat16))
    xb = bits(torch.from_numpy(x).to(torch.bfloat16))
    exact = np.zeros((4, 6), np.int64)
    for o in range(4):
        for i in range(6):
            exact[o, i] = sum(int(dy[t, o]) * int(x[t, i]) for t in range(16))
    np.testing.assert_array_equal(step.dw(dyb, xb), exact.astype(np.float32))


def test_dw_is_not_transposed():
    """dW[o, i] pairs column o of dY with column i of X (an outer product for T = 1)."""
    dy = bits(torch.tensor([[1.0, 2.0, 3.0]]).to(torch.bfloat16))
    x = bits(torch.tensor([[10.0, 20.0]]).to(torch.bfloat16))
    np.testing.assert_array_equal(step.dw(dy, x), np.array([[10, 20], [20, 40], [30, 60]], np.float32))


def test_sampled_positions_equal_dense():
    dy = bits(normal_bf16((64, 40), 1e-3, seed=3))
    x = bits(normal_bf16((64, 24), 1.0, seed=4))
    dense = step.dw(dy, x)
    rows = np.array([0, 5, 39, 17, 17])
    cols = np.array([0, 23, 7, 8, 9])
    np.testing.assert_array_equal(step.dw_at(dy, x, rows, cols), dense[rows, cols])

