"""Plant plausible mistakes in copies of the oracle (on the CPU) and check a pin catches each.

This shows the pins are sharp enough: a dropped term, a wrong sign, a swapped
hyperparameter or a transposed operand in the oracle makes some pin fail.
"""
import numpy as np
import pytest

from oracle import bf16, optim
from tests import test_oracle_optim as pins
from tests.helpers import bits
from workloads import normal_bf16


def _mutant(kind):
    def update(opt, g, w, m, v, hp, t):
        if kind == "adamw_no_bias_correction" and opt == "adamw":
            lr, b1, b2 = optim.binary32(hp.lr), optim.binary32(hp.beta1), optim.binary32(hp.beta2)
            eps, wd = optim.binary32(hp.eps), optim.binary32(hp.weight_decay)
            m1 = b1 * m + (1 - b1) * g
            v1 = b2 * v + (1 - b2) * g * g
            return w * (1 - lr * wd) - lr * m1 / (np.sqrt(v1) + eps), m1, v1
        if kind == "adamw_coupled_decay" and opt == "adamw":
            wd = optim.binary32(hp.weight_decay)
            hp0 = type(hp)(**{**hp.__dict__, "weight_decay": 0.0})
            return optim.update("adamw", g + wd * w, w, m, v, hp0, t)
        if kind == "sign_flip":
            w1, m1, v1 = optim.update(opt, g, w, m, v, hp, t)
            return 2 * w - w1, m1, v1
        if kind == "lion_beta2_in_sign" and opt == "lion":
            hp2 = type(hp)(**{**hp.__dict__, "beta1": hp.beta2})
            w1, _, _ = optim.update("lion", g, w, m, v, hp2, t)
            _, m1, _ = optim.update("lion", g, w, m, v, hp, t)
            return w1, m1, None
        if kind == "momentum_dampened" and opt == "sgd_momentum":
            mu = optim.binary32(hp.momentum)
            m1 = mu * m + (1 - mu) * (g + optim.binary32(hp.weight_decay) * w)
            return w - optim.binary32(hp.lr) * m1, m1, None
        if kind == "rmsprop_no_sqrt" and opt == "rmsprop":
            w1, m1, v1 = optim.update(opt, g, w, m, v, hp, t)
            lr, eps, wd = optim.binary32(hp.lr), optim.binary32(hp.eps), optim.binary32(hp.weight_decay)
            return w - lr * (g + wd * w) / (v1 + eps), m1, v1
        return optim.update(opt, g, w, m, v, hp, t)
    return update


def _all_pins(update):
    for p in pins.CLOSED_FORM_PINS:
        p(update)
    for opt in ["adamw", "nadam", "radam", "rmsprop", "adagrad", "sgd", "sgd_momentum"]:
        pins.pin_against_torch(update, opt, steps=4)


@pytest.mark.parametrize("kind", ["adamw_no_bias_correction", "adamw_coupled_decay", "sign_flip",
                                  "lion_beta2_in_sign", "momentum_dampened", "rmsprop_no_sqrt"])
def test_pins_catch_planted_optimizer_mistakes(kind):
    with pytest.raises(AssertionError):
        _all_pins(_mutant(kind))


def test_pins_pass_on_the_real_oracle():
    _all_pins(optim.update)


def test_transposed_gradient_is_caught():
    from tests.test_oracle_dw import _brute_force
    dy = bits(normal_bf16((9, 4), 1e-2, seed=11))
    x = bits(normal_bf16((9, 4), 1.0, seed=12))
    wrong = (bf16.to_f64(x).T @ bf16.to_f64(dy)).astype(np.float32)  # X^T dY instead of dY^T X
    with pytest.raises(AssertionError):
        np.testing.assert_allclose(wrong, _brute_force(dy, x), rtol=2 ** -23, atol=0)


def test_round_to_nearest_fails_the_sr_expectation_pin():
    x = np.float32(1.0 + 2.0 ** -9)
    out = bf16.to_f64(bf16.round_nearest_even(np.full(65536, x, np.float32)))
    assert out.sum() / 65536.0 != float(x)
