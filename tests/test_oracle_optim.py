"""Pins for the oracle's eight optimizers (CPU only).

Three kinds of pin, none of which retypes the oracle's formulas:
  * closed forms (step 1 from zero moments, zero gradient, Lion's unit step);
  * hand-worked examples whose intermediate values are written out below;
  * multi-step float64 cross-checks against ``torch.optim`` (an independent
    implementation) for the seven optimizers it ships.
The pin functions take the update routine as an argument so that
test_oracle_mutations.py can run them against planted mistakes.
"""
import math

import numpy as np
import pytest
import torch

from oracle import optim
from workloads import Hparams, default_hparams

F = np.float64


def _g(seed, n=4096, scale=1e-3):
    return np.random.default_rng(seed).standard_normal(n) * scale


# ----------------------------------------------------------------------------- closed forms

def pin_adamw_step1(update):
    g = _g(0)
    w = _g(1, scale=0.02)
    hp = Hparams(lr=1e-3, weight_decay=0.0)
    w1, m1, v1 = update("adamw", g, w, np.zeros_like(g), np.zeros_like(g), hp, 1)
    lr, eps = optim.binary32(1e-3), optim.binary32(1e-8)
    np.testing.assert_allclose(w1 - w, -lr * g / (np.abs(g) + eps), rtol=1e-9, atol=1e-15)
    # with decoupled weight decay the step-1 move is the decay plus the same sign step
    hp = Hparams(lr=1e-3, weight_decay=0.1)
    w1, _, _ = update("adamw", g, w, np.zeros_like(g), np.zeros_like(g), hp, 1)
    lam = optim.binary32(1e-3) * optim.binary32(0.1)
    np.testing.assert_allclose(w1, w * (1 - lam) - lr * g / (np.abs(g) + eps), rtol=1e-9, atol=1e-15)


def pin_adamw_zero_gradient(update):
    w = _g(2, scale=0.02)
    z = np.zeros_like(w)
    hp = Hparams(lr=1e-3, weight_decay=0.01)
    for t in (1, 7):
        w1, m1, v1 = update("adamw", z, w, z, z, hp, t)
        assert np.all(m1 == 0) and np.all(v1 == 0)
        np.testing.assert_array_equal(w1, w * (1 - optim.binary32(1e-3) * optim.binary32(0.01)))


def pin_adamw_hand_2x2(update):
    """beta1 = 1/2, beta2 = 3/4, lr = 1/10, eps = 0, wd = 1/2, t = 2.

    g = [[1, -2], [1/2, 0]], m = [[1/2, 0], [1, -1]], v = [[1/4, 1], [0, 4]], W = [[1, -1], [1/2, 2]]
    m' = m/2 + g/2             = [[3/4, -1], [3/4, -1/2]]
    v' = 3v/4 + g^2/4          = [[7/16, 7/4], [1/16, 3]]
    m^ = m'/(1 - 1/4)          = [[1, -4/3], [1, -2/3]]
    v^ = v'/(1 - 9/16)         = [[1, 4], [1/7, 48/7]]
    W(1 - lr wd) = 0.95 W      = [[0.95, -0.95], [0.475, 1.9]]
    lr m^/sqrt(v^)             = [[0.1, -0.0666667], [0.2645751, -0.0254588]]
    W'                         = [[0.85, -0.8833333], [0.2104249, 1.9254588]]
    """
    g = np.array([1, -2, 0.5, 0], F)
    m = np.array([0.5, 0, 1, -1], F)
    v = np.array([0.25, 1, 0, 4], F)
    w = np.array([1, -1, 0.5, 2], F)
    hp = Hparams(lr=0.1, beta1=0.5, beta2=0.75, eps=0.0, weight_decay=0.5)
    w1, m1, v1 = update("adamw", g, w, m, v, hp, 2)
    np.testing.assert_allclose(m1, [0.75, -1, 0.75, -0.5], rtol=1e-12)
    np.testing.assert_allclose(v1, [7 / 16, 7 / 4, 1 / 16, 3], rtol=1e-12)
    np.testing.assert_allclose(w1, [0.85, -0.8833333, 0.2104249, 1.9254588], rtol=2e-7, atol=1e-7)


def pin_lion(update):
    """c uses beta1, the moment update uses beta2; the step is exactly lr in magnitude."""
    hp = Hparams(lr=0.01, beta1=0.9, beta2=0.99, weight_decay=0.5)
    w = np.array([1.0, 1.0, -2.0, 0.5], F)
    m = np.array([1.0, 1.0, 0.0, 0.0], F)
    g = np.array([-9.5, -1.0, 3.0, 0.0], F)
    w1, m1, v1 = update("lion", g, w, m, None, hp, 3)
    assert v1 is None
    # c = 0.9 m + 0.1 g = [-0.05, 0.8, 0.3, 0] -> sign [-1, +1, +1, 0]
    lr, wd = optim.binary32(0.01), optim.binary32(0.5)
    np.testing.assert_allclose(w1, w * (1 - lr * wd) - lr * np.array([-1, 1, 1, 0]), rtol=1e-12)
    # m' = 0.99 m + 0.01 g = [0.895, 0.98, 0.03, 0]
    np.testing.assert_allclose(m1, [0.895, 0.98, 0.03, 0.0], rtol=1e-6, atol=1e-12)


def pin_rmsprop_adagrad_step1(update):
    g = _g(3)
    w = _g(4, scale=0.02)
    z = np.zeros_like(g)
    lr, eps = optim.binary32(1e-3), optim.binary32(1e-8)
    w1, m1, v1 = update("rmsprop", g, w, None, z, Hparams(lr=1e-3, weight_decay=0.0, alpha=0.99), 1)
    assert m1 is None
    np.testing.assert_allclose(w1 - w, -lr * g / (np.sqrt(1 - optim.binary32(0.99)) * np.abs(g) + eps), rtol=1e-9)
    w1, m1, v1 = update("adagrad", g, w, None, z, Hparams(lr=1e-3, weight_decay=0.0, eps=1e-10), 1)
    np.testing.assert_allclose(w1 - w, -lr * g / (np.abs(g) + optim.binary32(1e-10)), rtol=1e-9)
    np.testing.assert_allclose(v1, g * g, rtol=1e-15)


def pin_sgd(update):
    g, w = _g(5), _g(6, scale=0.02)
    hp = Hparams(lr=1e-2, weight_decay=0.1, momentum=0.9)
    lr, wd, mu = optim.binary32(1e-2), optim.binary32(0.1), optim.binary32(0.9)
    w1, m1, v1 = update("sgd", g, w, None, None, hp, 4)
    np.testing.assert_allclose(w1, w - lr * (g + wd * w), rtol=1e-14)
    m = _g(7)
    w1, m1, v1 = update("sgd_momentum", g, w, m, None, hp, 4)
    np.testing.assert_allclose(m1, mu * m + g + wd * w, rtol=1e-12, atol=1e-18)
    np.testing.assert_allclose(w1, w - lr * m1, rtol=1e-14)


def pin_radam_early_steps(update):
    """rho_1 = 1 for every beta2, so step 1 is an un-rectified SGD-with-momentum step: W - lr (g + wd W)."""
    rho_inf, rho_1 = optim.radam_rho(1, optim.binary32(0.999))
    assert abs(rho_1 - 1.0) < 1e-9
    g, w = _g(8), _g(9, scale=0.02)
    z = np.zeros_like(g)
    hp = Hparams(lr=1e-3, weight_decay=0.01)
    w1, _, _ = update("radam", g, w, z, z, hp, 1)
    lr, wd = optim.binary32(1e-3), optim.binary32(0.01)
    np.testing.assert_allclose(w1, w - lr * (g + wd * w), rtol=1e-9)


CLOSED_FORM_PINS = [pin_adamw_step1, pin_adamw_zero_gradient, pin_adamw_hand_2x2, pin_lion,
                    pin_rmsprop_adagrad_step1, pin_sgd, pin_radam_early_steps]


@pytest.mark.parametrize("pin", CLOSED_FORM_PINS, ids=lambda p: p.__name__)
def test_closed_forms(pin):
    pin(optim.update)


# ----------------------------------------------------------------------------- torch.optim

def _torch_optimizer(opt, p, hp):
    b32 = optim.binary32
    lr, wd = b32(hp.lr), b32(hp.weight_decay)
    betas = (b32(hp.beta1), b32(hp.beta2))
    if opt == "adamw":
        return torch.optim.AdamW([p], lr=lr, betas=betas, eps=b32(hp.eps), weight_decay=wd, foreach=False)
    if opt == "nadam":
        return torch.optim.NAdam([p], lr=lr, betas=betas, eps=b32(hp.eps), weight_decay=wd,
                                 momentum_decay=b32(hp.momentum_decay), foreach=False)
    if opt == "radam":
        return torch.optim.RAdam([p], lr=lr, betas=betas, eps=b32(hp.eps), weight_decay=wd, foreach=False)
    if opt == "rmsprop":
        return torch.optim.RMSprop([p], lr=lr, alpha=b32(hp.alpha), eps=b32(hp.eps), weight_decay=wd,
                                   foreach=False)
    if opt == "adagrad":
        return torch.optim.Adagrad([p], lr=lr, lr_decay=b32(hp.lr_decay), eps=b32(hp.eps),
                                   weight_decay=wd, foreach=False)
    if opt == "sgd":
        return torch.optim.SGD([p], lr=lr, weight_decay=wd, foreach=False)
    if opt == "sgd_momentum":
        return torch.optim.SGD([p], lr=lr, momentum=b32(hp.momentum), weight_decay=wd, foreach=False)
    raise ValueError(opt)


def pin_against_torch(update, opt, steps=10, hp=None):
    hp = hp or default_hparams(opt, lr=1e-3, weight_decay=0.05)
    n = 2048
    w0 = _g(10, n, 0.02)
    grads = [_g(100 + t, n, 1e-2 * (1 + t % 3)) for t in range(steps)]
    old = torch.get_default_dtype()
    torch.set_default_dtype(torch.float64)
    try:
        p = torch.nn.Parameter(torch.tensor(w0))
        topt = _torch_optimizer(opt, p, hp)
        for t in range(steps):
            p.grad = torch.tensor(grads[t])
            topt.step()
        st = topt.state[p]
    finally:
        torch.set_default_dtype(old)
    use_m, use_v = optim.USES[opt]
    w, m, v = w0.copy(), (np.zeros(n) if use_m else None), (np.zeros(n) if use_v else None)
    for t in range(steps):
        w, m, v = update(opt, grads[t], w, m, v, hp, t + 1)
    np.testing.assert_allclose(w, p.detach().numpy(), rtol=1e-11, atol=1e-15)
    mkey = {"adamw": "exp_avg", "nadam": "exp_avg", "radam": "exp_avg", "sgd_momentum": "momentum_buffer"}
    vkey = {"adamw": "exp_avg_sq", "nadam": "exp_avg_sq", "radam": "exp_avg_sq",
            "rmsprop": "square_avg", "adagrad": "sum"}
    if opt in mkey:
        np.testing.assert_allclose(m, st[mkey[opt]].numpy(), rtol=1e-11, atol=1e-18)
    if opt in vkey:
        np.testing.assert_allclose(v, st[vkey[opt]].numpy(), rtol=1e-11, atol=1e-20)


@pytest.mark.parametrize("opt", ["adamw", "nadam", "radam", "rmsprop", "adagrad", "sgd", "sgd_momentum"])
def test_against_torch_optim(opt):
    pin_against_torch(optim.update, opt)


def test_radam_rectified_branch_reached_and_matches_torch():
    rho = [optim.radam_rho(t, optim.binary32(0.999))[1] for t in range(1, 11)]
    assert rho[4] <= 5.0 < rho[5]  # t = 6 is the first rectified step with beta2 = 0.999
    pin_against_torch(optim.update, "radam", steps=12)


def test_adagrad_lr_decay_matches_torch():
    pin_against_torch(optim.update, "adagrad", steps=6, hp=Hparams(lr=1e-2, eps=1e-10, lr_decay=0.3,
                                                                   weight_decay=0.01))


def test_nadam_mu_product():
    b1, psi = optim.binary32(0.9), optim.binary32(4e-3)
    mus = [b1 * (1 - 0.5 * 0.96 ** (i * psi)) for i in range(1, 6)]
    assert math.isclose(optim.nadam_mu_product(5, b1, psi), math.prod(mus), rel_tol=1e-15)


def test_step_must_be_one_based():
    with pytest.raises(ValueError):
        optim.update("sgd", np.zeros(1), np.zeros(1), None, None, Hparams(), 0)
