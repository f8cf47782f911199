"""The eight element-wise optimizers, in float64, from their own published definitions.

FORGE summary, §3 Key contributions, "Generality", names AdamW, NAdam, RAdam,
Lion, RMSprop, AdaGrad, SGD and SGD-momentum as fully fused, but gives no
formulas.  Each update below is the optimizer's published definition, written
in the conventions of ``torch.optim`` (so the library routine can cross-check
it in float64):

* AdamW  -- Loshchilov & Hutter, "Decoupled Weight Decay Regularization" (ICLR'19), Alg. 2.
* NAdam  -- Dozat, "Incorporating Nesterov Momentum into Adam" (ICLR'16 workshop),
            with the momentum schedule mu_t = beta1 (1 - 0.5 * 0.96^(t psi)).
* RAdam  -- Liu et al., "On the Variance of the Adaptive Learning Rate and Beyond" (ICLR'20), Alg. 2.
* Lion   -- Chen et al., "Symbolic Discovery of Optimization Algorithms" (NeurIPS'23), Alg. 2.
* RMSprop-- Tieleman & Hinton, Coursera lecture 6.5 (no momentum, not centred).
* AdaGrad-- Duchi, Hazan & Singer, JMLR 12 (2011), diagonal form, with lr decay lr/(1+(t-1) decay).
* SGD, SGD-momentum (heavy ball, dampening 0, not Nesterov: m <- mu m + g).

Weight decay: decoupled (W <- W (1 - lr wd)) for AdamW and Lion, as their
definitions state; coupled L2 (g <- g + wd W) for the other six, as in their
original form.  The summary is silent on this; it is our reading.

``t`` is the 1-based step.  Every function is stateless: it takes the moments
before the step and returns them after it.  Bias corrections, the NAdam
momentum product and the RAdam rectification depend on ``t`` only, which
assumes the run started at t = 1 with the same hyperparameters.

Pinned by: closed forms at t = 1 and for g = 0, Lion's |sign| step, and
multi-step float64 cross-checks against ``torch.optim`` for the seven optimizers
it ships (tests/test_oracle_optim.py).
"""
from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

OPTIMIZERS = ("adamw", "nadam", "radam", "lion", "rmsprop", "adagrad", "sgd", "sgd_momentum")
USES = {  # (m, v)
    "adamw": (True, True), "nadam": (True, True), "radam": (True, True),
    "lion": (True, False), "sgd_momentum": (True, False),
    "rmsprop": (False, True), "adagrad": (False, True), "sgd": (False, False),
}


def binary32(x: float) -> float:
    """A hyperparameter as it crosses the C ABI: rounded to binary32."""
    return float(np.float32(x))


def nadam_mu(t: int, beta1: float, psi: float) -> float:
    return beta1 * (1.0 - 0.5 * 0.96 ** (t * psi))


def nadam_mu_product(t: int, beta1: float, psi: float) -> float:
    p = 1.0
    for i in range(1, t + 1):
        p *= nadam_mu(i, beta1, psi)
    return p


def radam_rho(t: int, beta2: float) -> Tuple[float, float]:
    """(rho_inf, rho_t) of the RAdam variance rectification."""
    rho_inf = 2.0 / (1.0 - beta2) - 1.0
    b2t = beta2 ** t
    return rho_inf, rho_inf - 2.0 * t * b2t / (1.0 - b2t)


def update(opt: str, g, w, m: Optional[np.ndarray], v: Optional[np.ndarray], hp, t: int):
    """One step of optimizer ``opt`` in float64.

    g, w, m, v: float64 arrays (gradient, weight, first and second moment before the
    step; m or v is None where ``opt`` does not use it).  ``hp`` has the fields of
    ``workloads.Hparams``; each is first rounded to binary32 as the ABI carries it.
    Returns (w_new, m_new, v_new) in float64.
    """
    if t < 1:
        raise ValueError("step t is 1-based")
    lr, b1, b2 = binary32(hp.lr), binary32(hp.beta1), binary32(hp.beta2)
    eps, wd = binary32(hp.eps), binary32(hp.weight_decay)
    g = np.asarray(g, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)

    if opt == "adamw":
        m1 = b1 * m + (1.0 - b1) * g
        v1 = b2 * v + (1.0 - b2) * g * g
        m_hat = m1 / (1.0 - b1 ** t)
        v_hat = v1 / (1.0 - b2 ** t)
        w1 = w * (1.0 - lr * wd) - lr * m_hat / (np.sqrt(v_hat) + eps)
        return w1, m1, v1

    if opt == "nadam":
        psi = binary32(hp.momentum_decay)
        gc = g + wd * w
        mu_t, mu_next = nadam_mu(t, b1, psi), nadam_mu(t + 1, b1, psi)
        prod_t = nadam_mu_product(t, b1, psi)
        m1 = b1 * m + (1.0 - b1) * gc
        v1 = b2 * v + (1.0 - b2) * gc * gc
        denom = np.sqrt(v1 / (1.0 - b2 ** t)) + eps
        w1 = (w - lr * (1.0 - mu_t) / (1.0 - prod_t) * gc / denom
              - lr * mu_next / (1.0 - prod_t * mu_next) * m1 / denom)
        return w1, m1, v1

    if opt == "radam":
        gc = g + wd * w
        m1 = b1 * m + (1.0 - b1) * gc
        v1 = b2 * v + (1.0 - b2) * gc * gc
        m_hat = m1 / (1.0 - b1 ** t)
        rho_inf, rho_t = radam_rho(t, b2)
        if rho_t > 5.0:
            r_t = math.sqrt((rho_t - 4.0) * (rho_t - 2.0) * rho_inf
                            / ((rho_inf - 4.0) * (rho_inf - 2.0) * rho_t))
            w1 = w - lr * m_hat * r_t * math.sqrt(1.0 - b2 ** t) / (np.sqrt(v1) + eps)
        else:
            w1 = w - lr * m_hat
        return w1, m1, v1

    if opt == "lion":
        c = b1 * m + (1.0 - b1) * g
        w1 = w * (1.0 - lr * wd) - lr * np.sign(c)
        m1 = b2 * m + (1.0 - b2) * g
        return w1, m1, None

    if opt == "rmsprop":
        alpha = binary32(hp.alpha)
        gc = g + wd * w
        v1 = alpha * v + (1.0 - alpha) * gc * gc
        w1 = w - lr * gc / (np.sqrt(v1) + eps)
        return w1, None, v1

    if opt == "adagrad":
        gc = g + wd * w
        v1 = v + gc * gc
        clr = lr / (1.0 + (t - 1) * binary32(hp.lr_decay))
        w1 = w - clr * gc / (np.sqrt(v1) + eps)
        return w1, None, v1

    if opt == "sgd":
        return w - lr * (g + wd * w), None, None

    if opt == "sgd_momentum":
        mu = binary32(hp.momentum)
        m1 = mu * m + (g + wd * w)
        return w - lr * m1, m1, None

    raise ValueError(f"unknown optimizer {opt!r}")
