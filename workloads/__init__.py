"""Seeded synthetic workloads for the fused weight-gradient + optimizer step.

This module only draws random tensors and names shapes and hyperparameters.
It holds none of the method's arithmetic (no gradient, no optimizer, no
rounding rule), so both the CPU oracle and the CUDA library can take their
inputs from it without sharing any computation.

Shapes follow the layer shapes the FORGE summary evaluates on ("FORGE: Fused
On-Register Gradient Elimination for Memory-Efficient LLM Training", §4
Experimental results: Llama-3.1-8B and the Qwen3 family).  No dataset and no
trained weights are used: every tensor is a seeded draw from the stated
distribution, made in float32 and cast to bfloat16 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import torch

# Optimizer names, in the order of the C-ABI enum.
OPTIMIZERS: Tuple[str, ...] = (
    "adamw", "nadam", "radam", "lion", "rmsprop", "adagrad", "sgd", "sgd_momentum",
)

# Which moment slots an optimizer uses: (m, v).
MOMENTS: Dict[str, Tuple[bool, bool]] = {
    "adamw": (True, True), "nadam": (True, True), "radam": (True, True),
    "lion": (True, False), "sgd_momentum": (True, False),
    "rmsprop": (False, True), "adagrad": (False, True),
    "sgd": (False, False),
}


@dataclasses.dataclass(frozen=True)
class Hparams:
    """Hyperparameters as they cross the C ABI (every field is a binary32)."""
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    momentum: float = 0.9        # SGD-momentum mu
    alpha: float = 0.99          # RMSprop smoothing constant
    momentum_decay: float = 4e-3  # NAdam psi
    lr_decay: float = 0.0        # AdaGrad


def default_hparams(opt: str, lr: float = 1e-4, weight_decay: float = 0.01) -> Hparams:
    """Each optimizer's customary defaults, with the sweep's lr and weight decay."""
    if opt == "lion":
        return Hparams(lr=lr, weight_decay=weight_decay, beta1=0.9, beta2=0.99)
    if opt == "adagrad":
        return Hparams(lr=lr, weight_decay=weight_decay, eps=1e-10)
    return Hparams(lr=lr, weight_decay=weight_decay)


@dataclasses.dataclass(frozen=True)
class Layer:
    name: str
    d_out: int
    d_in: int


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: Tuple[Layer, ...]
    T: int
    x_std: float
    dy_std: float
    w_std: float = 0.02
    m_init: str = "zero"      # "zero" | "absnormal:<std>"
    v_init: str = "zero"      # "zero" | "uniform:<hi>"
    steps: Tuple[int, ...] = (1,)
    description: str = ""

    def flops_per_step(self) -> int:
        return sum(2 * self.T * l.d_out * l.d_in for l in self.layers)

    def params(self) -> int:
        return sum(l.d_out * l.d_in for l in self.layers)


def _llama8b_mlp() -> Workload:
    return Workload(
        name="llama3.1-8b-mlp",
        layers=(Layer("gate", 14336, 4096), Layer("up", 14336, 4096), Layer("down", 4096, 14336)),
        T=4096, x_std=1.0, dy_std=1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6",
        steps=(10,),
        description="Llama-3.1-8B MLP weight updates (gate/up 14336x4096, down 4096x14336), "
                    "T=4096 tokens, AdamW with FP32 moments at step 10",
    )


def _qwen14b_sweep(n_layers: int = 40) -> Workload:
    per = (Layer("q", 5120, 5120), Layer("k", 1024, 5120), Layer("v", 1024, 5120),
           Layer("o", 5120, 5120), Layer("gate", 17408, 5120), Layer("up", 17408, 5120),
           Layer("down", 5120, 17408))
    layers = tuple(Layer(f"L{i}.{l.name}", l.d_out, l.d_in) for i in range(n_layers) for l in per)
    return Workload(
        name=f"qwen3-14b-linear-sweep-{n_layers}L", layers=layers, T=8192, x_std=1.0, dy_std=1e-3,
        m_init="absnormal:1e-4", v_init="uniform:1e-6", steps=(10,),
        description=f"Qwen3-14B-shaped backward linear sweep, {n_layers} layers x 7 projections, T=8192",
    )


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload(
        name="tiny", layers=(Layer("w", 512, 256),), T=256, x_std=1.0, dy_std=1e-2,
        steps=(1, 2, 3), description="single 512x256 layer, T=256, AdamW, 3 steps, fresh X/dY per step"),
    "llama8b-mlp": _llama8b_mlp(),
    "coverage-4096": Workload(
        name="coverage-4096", layers=(Layer("w", 4096, 4096),), T=8192, x_std=1.0, dy_std=1e-3,
        steps=(1, 2, 3, 4, 5), description="one 4096x4096 layer, T=8192, each optimizer, 5 steps, FP32 states"),
    "int8-4096": Workload(
        name="int8-4096", layers=(Layer("w", 4096, 4096),), T=2048, x_std=1.0, dy_std=1e-3,
        steps=(1,), description="one 4096x4096 layer, T=2048, AdamW with INT8 block-64 moments"),
    "qwen14b-sweep": _qwen14b_sweep(40),
    # the Llama MLP's token count and distributions on one square layer: a case small enough for a
    # full profiler capture that keeps the Llama layers' balance of mainloop and epilogue
    "sq4096-t4096": Workload(
        name="sq4096-t4096", layers=(Layer("w", 4096, 4096),), T=4096, x_std=1.0, dy_std=1e-3,
        m_init="absnormal:1e-4", v_init="uniform:1e-6", steps=(10,),
        description="one 4096x4096 layer, T=4096, AdamW with FP32 moments at step 10 (Llama MLP balance)"),
}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & ((1 << 63) - 1))
    return g


def normal_bf16(shape: Sequence[int], std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in float32, cast to bfloat16 (round-to-nearest-even)."""
    t = torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return (t * std).to(torch.bfloat16)


def moment_init(kind: str, shape: Sequence[int], seed: int, device="cpu") -> torch.Tensor:
    """Initial FP32 moment: 'zero', 'absnormal:<std>' (|N(0,std^2)|) or 'uniform:<hi>' (U(0,hi))."""
    if kind == "zero":
        return torch.zeros(*shape, dtype=torch.float32, device=device)
    name, _, arg = kind.partition(":")
    val = float(arg)
    if name == "absnormal":
        return torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32).abs_() * val
    if name == "uniform":
        return torch.rand(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32) * val
    raise ValueError(f"unknown moment init {kind!r}")


def layer_seed(base: int, layer_index: int, what: str, step: int = 0) -> int:
    """Deterministic per-(layer, tensor, step) seed so every draw is reproducible alone."""
    tag = {"x": 1, "dy": 2, "w": 3, "m": 4, "v": 5}[what]
    return (base * 1_000_003 + layer_index * 7919 + tag * 104_729 + step * 15_485_863) & ((1 << 62) - 1)


def activations(wl: Workload, layer_index: int, step: int, seed: int = 0, device="cpu",
                ) -> Tuple[torch.Tensor, torch.Tensor]:
    """(dY [T, d_out], X [T, d_in]) in bfloat16, both token-major (row-major)."""
    l = wl.layers[layer_index]
    dy = normal_bf16((wl.T, l.d_out), wl.dy_std, layer_seed(seed, layer_index, "dy", step), device)
    x = normal_bf16((wl.T, l.d_in), wl.x_std, layer_seed(seed, layer_index, "x", step), device)
    return dy, x


def layer_state(wl: Workload, layer_index: int, opt: str = "adamw", seed: int = 0, device="cpu",
                ) -> Tuple[torch.Tensor, Optional[torch.Tensor], Optional[torch.Tensor]]:
    """(W [d_out, d_in] bf16, m or None, v or None) FP32 initial optimizer state."""
    l = wl.layers[layer_index]
    w = normal_bf16((l.d_out, l.d_in), wl.w_std, layer_seed(seed, layer_index, "w"), device)
    use_m, use_v = MOMENTS[opt]
    m = moment_init(wl.m_init, (l.d_out, l.d_in), layer_seed(seed, layer_index, "m"), device) if use_m else None
    v = moment_init(wl.v_init, (l.d_out, l.d_in), layer_seed(seed, layer_index, "v"), device) if use_v else None
    return w, m, v


def random_codes(shape: Sequence[int], seed: int, lo: int, hi: int) -> torch.Tensor:
    """Uniform int8 codes in [lo, hi] (for INT8 state tests)."""
    return torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed), dtype=torch.int8)


def positive_scales(n: int, seed: int, hi: float) -> torch.Tensor:
    """Per-block FP32 scales drawn from U(0, hi) (for INT8 state tests)."""
    return torch.rand(n, generator=_gen(seed), dtype=torch.float32) * hi


def sample_positions(d_out: int, d_in: int, n: int, seed: int, block: int = 1) -> Tuple[List[int], List[int]]:
    """n distinct (row, col) positions, col a multiple of `block` (start of a block)."""
    g = _gen(seed)
    total = d_out * (d_in // block)
    n = min(n, total)
    flat = torch.randperm(total, generator=g)[:n].sort().values
    rows = (flat // (d_in // block)).tolist()
    cols = ((flat % (d_in // block)) * block).tolist()
    return rows, cols


def fp8_e4m3(t: torch.Tensor) -> Tuple[torch.Tensor, float]:
    """Per-tensor E4M3 codes of a float32 tensor, as an FP8 training recipe hands them over:
    scale = amax / 448 (the largest E4M3 magnitude), codes = PyTorch's float8_e4m3fn cast of t / scale.
    Returns (uint8 codes, scale)."""
    t = t.float()
    amax = float(t.abs().max()) if t.numel() else 0.0
    scale = float(torch.tensor(amax / 448.0 if amax > 0 else 1.0, dtype=torch.float32))
    codes = (t / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def activations_fp8(wl: Workload, layer_index: int, step: int, seed: int = 0, device="cpu", per_channel=False):
    """(dY codes [T, d_out], s_dY, X codes [T, d_in], s_X): the layer's activations drawn as for
    ``activations`` (float32, same seeds) and quantised to E4M3 per tensor (float scales) or, with
    ``per_channel``, per column (float32 scale vectors on `device`)."""
    l = wl.layers[layer_index]
    dy = torch.randn(wl.T, l.d_out, generator=_gen(layer_seed(seed, layer_index, "dy", step), device),
                     device=device) * wl.dy_std
    x = torch.randn(wl.T, l.d_in, generator=_gen(layer_seed(seed, layer_index, "x", step), device),
                    device=device) * wl.x_std
    if per_channel:
        dyq, s_dy = fp8_e4m3_channels(dy)
        xq, s_x = fp8_e4m3_channels(x)
    else:
        dyq, s_dy = fp8_e4m3(dy)
        xq, s_x = fp8_e4m3(x)
    return dyq, s_dy, xq, s_x


def fp8_e4m3_channels(t: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-column E4M3 codes of a float32 [rows, cols] tensor: scale[c] = amax(|t[:, c]|) / 448
    (1 for an all-zero column), codes = PyTorch's float8_e4m3fn cast of t / scale.
    Returns (uint8 codes, float32 scales [cols])."""
    t = t.float()
    amax = t.abs().amax(dim=0) if t.numel() else torch.zeros(t.shape[1])
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).float()
    codes = (t / scale[None, :]).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale
