"""A linear layer whose backward is the fused step: PyTorch autograd integration.

`ForgeLinear` computes y = x W^T.  Its backward does for one linear layer what the FORGE method
does in a training step ("FORGE: Fused On-Register Gradient Elimination for Memory-Efficient LLM
Training", §2 Methodology, Core mechanism): the input gradient dX = dY W is taken from the weights
as they were, then the weight gradient dW = dY^T X is accumulated tile by tile and consumed by the
optimizer inside the same kernel, which updates W and the optimizer state in place
(`linear_backward`).  No weight gradient exists afterwards: `weight.grad` stays None and there is
no separate optimizer step.

The forward is PyTorch's own `linear`; the backward runs only this library's kernels.  Because the
weights change during the backward, a weight that the same backward reads again (tied weights, a
layer applied twice in one step) cannot be trained this way, and gradient accumulation over
micro-batches becomes one optimizer step per micro-batch.  The layer refuses a second backward for
one forward.
"""
from __future__ import annotations

from typing import Any, Optional

import torch

from . import fused_dw_step, linear_backward

__all__ = ["ForgeLinear"]

# moment slots (m, v) each optimizer keeps
_MOMENTS = {
    "adamw": (True, True), "nadam": (True, True), "radam": (True, True),
    "lion": (True, False), "sgd_momentum": (True, False),
    "rmsprop": (False, True), "adagrad": (False, True),
    "sgd": (False, False),
}
_STATE_DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16, "int8": torch.int8}


class _ForgeLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, layer, want_dx):
        ctx.save_for_backward(x)
        ctx.layer, ctx.want_dx = layer, want_dx
        return torch.nn.functional.linear(x, weight)

    @staticmethod
    def backward(ctx, grad_out):
        (x,) = ctx.saved_tensors
        dY = grad_out.reshape(-1, grad_out.shape[-1]).to(torch.bfloat16).contiguous()
        X = x.reshape(-1, x.shape[-1]).contiguous()
        dX = torch.empty_like(X) if ctx.want_dx else None
        ctx.layer._step_once(dY, X, dX)
        return (None if dX is None else dX.reshape(x.shape)), None, None, None


class ForgeLinear(torch.nn.Module):
    """y = x W^T with W [out_features, in_features] bf16, trained by the fused backward.

    opt: one of adamw, nadam, radam, lion, rmsprop, adagrad, sgd, sgd_momentum.  hp: an object or
    dict with the nine hyperparameter fields (lr, beta1, beta2, eps, weight_decay, momentum, alpha,
    momentum_decay, lr_decay); missing fields take the library's defaults.  state: "fp32", "bf16"
    (stochastically rounded) or "int8" (codes with one scale per 64 elements; in_features a multiple
    of 64) moments.  seed: this layer's stochastic-rounding seed, distinct per layer.  `step` is the
    optimizer step the next backward takes; it starts at 1."""

    def __init__(self, in_features: int, out_features: int, opt: str = "adamw", hp: Any = None,
                 state: str = "fp32", seed: int = 0, device=None, init_std: float = 0.02):
        super().__init__()
        if opt not in _MOMENTS:
            raise ValueError(f"unknown optimizer {opt!r}")
        if state not in _STATE_DTYPES:
            raise ValueError("state: 'fp32', 'bf16' or 'int8'")
        dev = torch.device("cuda") if device is None else torch.device(device)
        w = torch.randn(out_features, in_features, device=dev) * init_std
        # the backward itself updates the weight: autograd gives it no gradient
        self.weight = torch.nn.Parameter(w.to(torch.bfloat16), requires_grad=False)
        use_m, use_v = _MOMENTS[opt]
        sdt = _STATE_DTYPES[state]
        shape = (out_features, in_features)
        self.register_buffer("m", torch.zeros(shape, dtype=sdt, device=dev) if use_m else None)
        self.register_buffer("v", torch.zeros(shape, dtype=sdt, device=dev) if use_v else None)
        q = state == "int8" and (use_m or use_v)
        # all-zero codes decode to zero whatever their scale
        self.register_buffer("qscales", torch.zeros(2 * out_features * in_features // 64, device=dev) if q else None)
        self.opt, self.hp, self.seed = opt, hp, int(seed)
        self.step = 1
        self._pending: Optional[int] = None

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        if x.dtype != torch.bfloat16:
            raise TypeError("ForgeLinear takes bfloat16 inputs")
        if not torch.is_grad_enabled():
            return torch.nn.functional.linear(x, self.weight)
        want_dx = x.requires_grad
        # autograd calls a backward only for outputs that depend on a tensor requiring grad
        anchor = x if want_dx else x.detach().requires_grad_(True)
        self._pending = self.step
        return _ForgeLinearFn.apply(anchor, self.weight, self, want_dx)

    def _step_once(self, dY, X, dX) -> None:
        if self._pending != self.step:
            raise RuntimeError("ForgeLinear: one backward per forward (the weights were already updated)")
        args = (self.weight.data, self.m, self.v, self.qscales)
        if dX is None:
            fused_dw_step(dY, X, *args, self.opt, self.hp, self.step, self.seed)
        else:
            linear_backward(dY, X, *args, dX, self.opt, self.hp, self.step, self.seed)
        self._pending = None
        self.step += 1

    def extra_repr(self) -> str:
        o, i = self.weight.shape
        state = "none" if self.m is None and self.v is None else str((self.m if self.m is not None else self.v).dtype)
        return f"in_features={i}, out_features={o}, opt={self.opt}, state={state}, step={self.step}"
