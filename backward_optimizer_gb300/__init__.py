"""Python binding of libforge.so, the fused weight-gradient + optimizer-step library.

The binding only marshals arguments: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  If the
library has not been built, every call raises ``ForgeUnavailable``: there is no
fallback path.

Entry points (same names as the C ABI in include/forge.h):
  fused_dw_step(dY, X, W, m, v, qscales, opt, hp, step, seed, stream=None)
  fused_dw_step_layers([(dY, X, W, m, v, qscales, seed), ...], opt, hp, step, stream=None)
  dw_gemm(dY, X, dW, stream=None)
  dx_gemm(dY, W, dX, stream=None)
  fused_dw_step_e4m3(dY8, X8, dy_scale, x_scale, W, m, v, qscales, opt, hp, step, seed, stream=None)
  dw_gemm_e4m3(dY8, X8, dy_scale, x_scale, dW, stream=None)
  linear_backward(dY, X, W, m, v, qscales, dX, opt, hp, step, seed, stream=None)
  opt_step(dW, W, m, v, qscales, opt, hp, step, seed, stream=None)
  sync_status(stream=None), set_wait_limit_ns(ns), launch_count()
"""
from __future__ import annotations

import ctypes
import os
from typing import Any, Optional

__all__ = [
    "OPT_KINDS", "STATE_FP32", "STATE_INT8_B64", "STATE_BF16", "ForgeError", "ForgeUnavailable", "lib", "library_path",
    "fused_dw_step", "fused_dw_step_layers", "dw_gemm", "dx_gemm", "linear_backward", "opt_step", "fused_dw_step_e4m3", "dw_gemm_e4m3", "sync_status", "set_wait_limit_ns", "launch_count", "build",
    "ForgeShape", "ForgeHparams", "hparams_struct",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libforge.so")

OPT_KINDS = {"adamw": 0, "nadam": 1, "radam": 2, "lion": 3, "rmsprop": 4, "adagrad": 5, "sgd": 6,
             "sgd_momentum": 7}
STATE_FP32 = 0
STATE_INT8_B64 = 1
STATE_BF16 = 2
STATUS = {0: "FORGE_OK", 1: "FORGE_ERR_INVALID_ARGUMENT", 2: "FORGE_ERR_UNSUPPORTED", 3: "FORGE_ERR_MISALIGNED",
          4: "FORGE_ERR_CUDA", 5: "FORGE_ERR_NOT_SM103", 6: "FORGE_ERR_TIMEOUT"}


class ForgeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class ForgeUnavailable(RuntimeError):
    pass


class ForgeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d_out", ctypes.c_int64), ("d_in", ctypes.c_int64),
                ("state", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class ForgeLayer(ctypes.Structure):
    _fields_ = [("dY", ctypes.c_void_p), ("X", ctypes.c_void_p), ("W", ctypes.c_void_p), ("m", ctypes.c_void_p),
                ("v", ctypes.c_void_p), ("qscales", ctypes.c_void_p), ("T", ctypes.c_int64), ("d_out", ctypes.c_int64),
                ("d_in", ctypes.c_int64), ("seed", ctypes.c_uint64)]


class ForgeHparams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in
                ("lr", "beta1", "beta2", "eps", "weight_decay", "momentum", "alpha", "momentum_decay", "lr_decay")]


_HP_DEFAULTS = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, momentum=0.9, alpha=0.99,
                    momentum_decay=4e-3, lr_decay=0.0)

_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    """Compile libforge.so in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library, with argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ForgeUnavailable(f"{_LIB_PATH} is not built; run backward_optimizer_gb300.build() first")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
    L.forge_fused_dw_step.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.POINTER(ForgeHparams),
                                      ctypes.POINTER(ForgeShape), i64, u64, vp]
    L.forge_fused_dw_step.restype = ctypes.c_int
    L.forge_fused_dw_step_layers.argtypes = [ctypes.POINTER(ForgeLayer), ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
                                             ctypes.POINTER(ForgeHparams), i64, vp]
    L.forge_fused_dw_step_layers.restype = ctypes.c_int
    L.forge_dw_gemm.argtypes = [vp, vp, vp, ctypes.POINTER(ForgeShape), vp]
    L.forge_dw_gemm.restype = ctypes.c_int
    f32 = ctypes.c_float
    L.forge_fused_dw_step_e4m3.argtypes = [vp, vp, f32, f32, vp, vp, vp, vp, ctypes.c_int,
                                           ctypes.POINTER(ForgeHparams), ctypes.POINTER(ForgeShape), i64, u64, vp]
    L.forge_fused_dw_step_e4m3.restype = ctypes.c_int
    L.forge_dw_gemm_e4m3.argtypes = [vp, vp, f32, f32, vp, ctypes.POINTER(ForgeShape), vp]
    L.forge_dw_gemm_e4m3.restype = ctypes.c_int
    L.forge_fused_dw_step_e4m3_channels.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                                    ctypes.POINTER(ForgeHparams), ctypes.POINTER(ForgeShape), i64,
                                                    u64, vp]
    L.forge_fused_dw_step_e4m3_channels.restype = ctypes.c_int
    L.forge_dw_gemm_e4m3_channels.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(ForgeShape), vp]
    L.forge_dw_gemm_e4m3_channels.restype = ctypes.c_int
    L.forge_dx_gemm.argtypes = [vp, vp, vp, ctypes.POINTER(ForgeShape), vp]
    L.forge_dx_gemm.restype = ctypes.c_int
    L.forge_linear_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.POINTER(ForgeHparams),
                                        ctypes.POINTER(ForgeShape), i64, u64, vp]
    L.forge_linear_backward.restype = ctypes.c_int
    L.forge_opt_step.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.POINTER(ForgeHparams),
                                 ctypes.POINTER(ForgeShape), i64, u64, vp]
    L.forge_opt_step.restype = ctypes.c_int
    L.forge_sync_status.argtypes = [vp]
    L.forge_sync_status.restype = ctypes.c_int
    L.forge_set_wait_limit_ns.argtypes = [u64]
    L.forge_set_wait_limit_ns.restype = None
    L.forge_debug_withhold_next_stage.argtypes = []
    L.forge_debug_withhold_next_stage.restype = None
    i32p = ctypes.POINTER(ctypes.c_int32)
    L.forge_launch_shape.argtypes = [ctypes.POINTER(ForgeShape), i32p, i32p, i32p, i32p]
    L.forge_launch_shape.restype = ctypes.c_int
    L.forge_dx_launch_shape.argtypes = [ctypes.POINTER(ForgeShape), i32p, i32p, i32p, i32p]
    L.forge_dx_launch_shape.restype = ctypes.c_int
    L.forge_launch_count.argtypes = []
    L.forge_launch_count.restype = u64
    L.forge_status_string.argtypes = [ctypes.c_int]
    L.forge_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def hparams_struct(hp: Any = None, **overrides) -> ForgeHparams:
    """A ForgeHparams from an object with the nine fields, a dict, or defaults + overrides."""
    vals = dict(_HP_DEFAULTS)
    if hp is not None:
        for k in _HP_DEFAULTS:
            if isinstance(hp, dict):
                if k in hp:
                    vals[k] = hp[k]
            elif hasattr(hp, k):
                vals[k] = getattr(hp, k)
    vals.update(overrides)
    return ForgeHparams(**{k: float(v) for k, v in vals.items()})


_HP_CACHE: dict = {}


def _hp_arg(hp: Any):
    """ctypes reference to the ForgeHparams of `hp`.  Immutable hyperparameter objects whose hash
    follows their values (a frozen dataclass such as workloads.Hparams, a tuple, None) are converted
    once and the struct is reused by later calls; anything else (a dict, an object whose fields a
    schedule may change between steps) is converted on every call.  The library copies what it
    needs during the call and keeps no pointer."""
    import dataclasses
    frozen = hp is None or isinstance(hp, tuple) or (
        dataclasses.is_dataclass(hp) and not isinstance(hp, type) and hp.__dataclass_params__.frozen)
    if not frozen:
        return ctypes.byref(hparams_struct(hp))
    hs = _HP_CACHE.get(hp)
    if hs is None:
        if len(_HP_CACHE) >= 256:
            _HP_CACHE.clear()
        hs = _HP_CACHE[hp] = hparams_struct(hp)
    return ctypes.byref(hs)


# ------------------------------------------------------------------ torch-facing wrappers

def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous (row-major)")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _expect(t, dtypes, shape, name: str) -> None:
    """Argument check before anything reaches the library: dtype among `dtypes`, exact shape."""
    if t is None:
        return
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected one of {[str(d) for d in dtypes]}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _state_args(W, m, v, qscales) -> None:
    import torch
    states = [t for t in (m, v) if t is not None]
    if len({t.dtype for t in states}) > 1:
        raise TypeError("m and v must share one state dtype")
    for t, name in ((m, "m"), (v, "v")):
        _expect(t, (torch.float32, torch.int8, torch.bfloat16), W.shape, name)
    if states and states[0].dtype == torch.int8:
        if qscales is None:
            raise ValueError("INT8 states need qscales")
        _expect(qscales, (torch.float32,), (2 * W.numel() // 64,), "qscales")


def _check(status: int, what: str) -> None:
    if status != 0:
        raise ForgeError(status, what)


def _shape(T: int, d_out: int, d_in: int, state: int) -> ForgeShape:
    return ForgeShape(T=int(T), d_out=int(d_out), d_in=int(d_in), state=int(state), reserved=0)


def _state_of(m, v) -> int:
    import torch
    for t in (m, v):
        if t is not None:
            if t.dtype == torch.int8:
                return STATE_INT8_B64
            return STATE_BF16 if t.dtype == torch.bfloat16 else STATE_FP32
    return STATE_FP32


def fused_dw_step(dY, X, W, m=None, v=None, qscales=None, opt: str = "adamw", hp: Any = None, step: int = 1,
                  seed: int = 0, stream=None) -> None:
    """One fused step on torch tensors: dY [T, d_out] bf16, X [T, d_in] bf16, W [d_out, d_in] bf16,
    m/v FP32, int8 or bf16 [d_out, d_in] (the dtype picks the state format), qscales FP32
    [2 * d_out * d_in / 64] for int8 states."""
    import torch
    T, d_out = dY.shape
    d_in = X.shape[1]
    for t, name, shp in ((dY, "dY", (T, d_out)), (X, "X", (T, d_in)), (W, "W", (d_out, d_in))):
        _expect(t, (torch.bfloat16,), shp, name)
    _state_args(W, m, v, qscales)
    shape = _shape(T, d_out, d_in, _state_of(m, v))
    st = lib().forge_fused_dw_step(_ptr(dY), _ptr(X), _ptr(W), _ptr(m), _ptr(v), _ptr(qscales), OPT_KINDS[opt],
                                   _hp_arg(hp), ctypes.byref(shape), int(step),
                                   int(seed) & (2**64 - 1), _stream(stream))
    _check(st, "forge_fused_dw_step")


def fused_dw_step_layers(layers, opt: str = "adamw", hp: Any = None, step: int = 1, stream=None) -> None:
    """The fused step for several independent layers in one call (up to 16 per kernel launch when
    their tiles are CTA pairs): `layers` is a sequence of (dY, X, W, m, v, qscales, seed), each as
    fused_dw_step takes them, all with the same state format.  Results equal per-layer
    fused_dw_step calls bit for bit."""
    import torch
    n = len(layers)
    arr = (ForgeLayer * max(n, 1))()
    state = None
    for i, (dY, X, W, m, v, qscales, seed) in enumerate(layers):
        T, d_out = dY.shape
        d_in = X.shape[1]
        for t, name, shp in ((dY, "dY", (T, d_out)), (X, "X", (T, d_in)), (W, "W", (d_out, d_in))):
            _expect(t, (torch.bfloat16,), shp, f"layers[{i}].{name}")
        _state_args(W, m, v, qscales)
        st = _state_of(m, v)
        if state is not None and st != state:
            raise TypeError("every layer must use the same state format")
        state = st
        arr[i] = ForgeLayer(_ptr(dY), _ptr(X), _ptr(W), _ptr(m), _ptr(v), _ptr(qscales), int(T), int(d_out), int(d_in),
                            int(seed) & (2**64 - 1))
    st = lib().forge_fused_dw_step_layers(arr, n, STATE_FP32 if state is None else state, OPT_KINDS[opt], _hp_arg(hp),
                                          int(step), _stream(stream))
    _check(st, "forge_fused_dw_step_layers")


def dw_gemm(dY, X, dW, stream=None) -> None:
    """dW [d_out, d_in] FP32 = dY^T X (the unfused baseline's gradient pass)."""
    import torch
    T, d_out = dY.shape
    _expect(dY, (torch.bfloat16,), (T, d_out), "dY")
    _expect(X, (torch.bfloat16,), (T, X.shape[1]), "X")
    _expect(dW, (torch.float32,), (d_out, X.shape[1]), "dW")
    shape = _shape(T, d_out, X.shape[1], STATE_FP32)
    _check(lib().forge_dw_gemm(_ptr(dY), _ptr(X), _ptr(dW), ctypes.byref(shape), _stream(stream)), "forge_dw_gemm")


def _channel_scales(dy_scale, x_scale, d_out: int, d_in: int) -> bool:
    """True for per-channel scales (two FP32 device vectors), False for two per-tensor floats."""
    import torch
    vec = isinstance(dy_scale, torch.Tensor), isinstance(x_scale, torch.Tensor)
    if vec[0] != vec[1]:
        raise TypeError("dy_scale and x_scale: both floats (per tensor) or both tensors (per channel)")
    if vec[0]:
        _expect(dy_scale, (torch.float32,), (d_out,), "dy_scale")
        _expect(x_scale, (torch.float32,), (d_in,), "x_scale")
    return vec[0]


def fused_dw_step_e4m3(dY, X, dy_scale, x_scale, W, m=None, v=None, qscales=None, opt: str = "adamw",
                       hp: Any = None, step: int = 1, seed: int = 0, stream=None) -> None:
    """The fused step with E4M3 operands: dY [T, d_out] and X [T, d_in] one-byte codes (uint8 or
    float8_e4m3fn tensors) with per-tensor scales (floats) or per-channel scales (FP32 device
    vectors of d_out and d_in); everything else as fused_dw_step."""
    import torch
    T, d_out = dY.shape
    d_in = X.shape[1]
    codes = (torch.uint8, torch.float8_e4m3fn)
    _expect(dY, codes, (T, d_out), "dY")
    _expect(X, codes, (T, d_in), "X")
    _expect(W, (torch.bfloat16,), (d_out, d_in), "W")
    _state_args(W, m, v, qscales)
    shape = _shape(T, d_out, d_in, _state_of(m, v))
    if _channel_scales(dy_scale, x_scale, d_out, d_in):
        st = lib().forge_fused_dw_step_e4m3_channels(
            _ptr(dY), _ptr(X), _ptr(dy_scale), _ptr(x_scale), _ptr(W), _ptr(m), _ptr(v), _ptr(qscales), OPT_KINDS[opt],
            _hp_arg(hp), ctypes.byref(shape), int(step), int(seed) & (2**64 - 1), _stream(stream))
        _check(st, "forge_fused_dw_step_e4m3_channels")
        return
    st = lib().forge_fused_dw_step_e4m3(_ptr(dY), _ptr(X), float(dy_scale), float(x_scale), _ptr(W), _ptr(m),
                                        _ptr(v), _ptr(qscales), OPT_KINDS[opt], _hp_arg(hp),
                                        ctypes.byref(shape), int(step), int(seed) & (2**64 - 1), _stream(stream))
    _check(st, "forge_fused_dw_step_e4m3")


def dw_gemm_e4m3(dY, X, dy_scale, x_scale, dW, stream=None) -> None:
    """dW [d_out, d_in] FP32 = dy_scale * x_scale * (dY^T X) from E4M3 codes (scales per tensor, or
    per channel as FP32 device vectors of d_out and d_in)."""
    import torch
    T, d_out = dY.shape
    codes = (torch.uint8, torch.float8_e4m3fn)
    _expect(dY, codes, (T, d_out), "dY")
    _expect(X, codes, (T, X.shape[1]), "X")
    _expect(dW, (torch.float32,), (d_out, X.shape[1]), "dW")
    shape = _shape(T, d_out, X.shape[1], STATE_FP32)
    if _channel_scales(dy_scale, x_scale, d_out, X.shape[1]):
        _check(lib().forge_dw_gemm_e4m3_channels(_ptr(dY), _ptr(X), _ptr(dy_scale), _ptr(x_scale), _ptr(dW),
                                                 ctypes.byref(shape), _stream(stream)), "forge_dw_gemm_e4m3_channels")
        return
    _check(lib().forge_dw_gemm_e4m3(_ptr(dY), _ptr(X), float(dy_scale), float(x_scale), _ptr(dW), ctypes.byref(shape),
                                    _stream(stream)), "forge_dw_gemm_e4m3")


def dx_gemm(dY, W, dX, stream=None) -> None:
    """dX [T, d_in] bf16 = dY W, the layer's input gradient (read W before any step replaces it)."""
    import torch
    T, d_out = dY.shape
    _expect(dY, (torch.bfloat16,), (T, d_out), "dY")
    _expect(W, (torch.bfloat16,), (d_out, W.shape[1]), "W")
    _expect(dX, (torch.bfloat16,), (T, W.shape[1]), "dX")
    shape = _shape(T, d_out, W.shape[1], STATE_FP32)
    _check(lib().forge_dx_gemm(_ptr(dY), _ptr(W), _ptr(dX), ctypes.byref(shape), _stream(stream)), "forge_dx_gemm")


def linear_backward(dY, X, W, m=None, v=None, qscales=None, dX=None, opt: str = "adamw", hp: Any = None,
                    step: int = 1, seed: int = 0, stream=None) -> None:
    """The linear layer's backward with the fused weight step: dX = dY W from the weights before the
    step, then the fused step, on one stream in that order."""
    import torch
    T, d_out = dY.shape
    d_in = X.shape[1]
    for t, name, shp in ((dY, "dY", (T, d_out)), (X, "X", (T, d_in)), (W, "W", (d_out, d_in)), (dX, "dX", (T, d_in))):
        _expect(t, (torch.bfloat16,), shp, name)
    _state_args(W, m, v, qscales)
    shape = _shape(T, d_out, d_in, _state_of(m, v))
    st = lib().forge_linear_backward(_ptr(dY), _ptr(X), _ptr(W), _ptr(m), _ptr(v), _ptr(qscales), _ptr(dX),
                                     OPT_KINDS[opt], _hp_arg(hp), ctypes.byref(shape),
                                     int(step), int(seed) & (2**64 - 1), _stream(stream))
    _check(st, "forge_linear_backward")


def opt_step(dW, W, m=None, v=None, qscales=None, opt: str = "adamw", hp: Any = None, step: int = 1, seed: int = 0,
             stream=None) -> None:
    """The unfused baseline's optimizer pass over a materialised FP32 gradient (None = zero gradient)."""
    import torch
    d_out, d_in = W.shape
    _expect(W, (torch.bfloat16,), (d_out, d_in), "W")
    _expect(dW, (torch.float32,), (d_out, d_in), "dW")
    _state_args(W, m, v, qscales)
    shape = _shape(0, d_out, d_in, _state_of(m, v))
    st = lib().forge_opt_step(_ptr(dW), _ptr(W), _ptr(m), _ptr(v), _ptr(qscales), OPT_KINDS[opt],
                              _hp_arg(hp), ctypes.byref(shape), int(step),
                              int(seed) & (2**64 - 1), _stream(stream))
    _check(st, "forge_opt_step")


def sync_status(stream=None) -> int:
    """Wait for the stream; return the device status (0, or 6 = a bounded wait ran out)."""
    return int(lib().forge_sync_status(_stream(stream)))


def set_wait_limit_ns(ns: int) -> None:
    lib().forge_set_wait_limit_ns(int(ns))


def launch_count() -> int:
    return int(lib().forge_launch_count())


def launch_shape(d_out: int, d_in: int, T: int = 64) -> dict:
    """Tile rows x columns, cluster size and CTA count the fused step uses for a layer."""
    vals = [ctypes.c_int32() for _ in range(4)]
    _check(lib().forge_launch_shape(ctypes.byref(_shape(T, d_out, d_in, STATE_FP32)), *[ctypes.byref(v) for v in vals]),
           "forge_launch_shape")
    return dict(zip(("tile_rows", "tile_cols", "cluster", "ctas"), (v.value for v in vals)))


def dx_launch_shape(T: int, d_out: int, d_in: int) -> dict:
    """Tile tokens x columns, cluster size and CTA count dx_gemm uses for a layer."""
    vals = [ctypes.c_int32() for _ in range(4)]
    _check(lib().forge_dx_launch_shape(ctypes.byref(_shape(T, d_out, d_in, STATE_FP32)),
                                       *[ctypes.byref(v) for v in vals]), "forge_dx_launch_shape")
    return dict(zip(("tile_rows", "tile_cols", "cluster", "ctas"), (v.value for v in vals)))


def debug_withhold_next_stage() -> None:
    """Test switch: the next tile-kernel launch withholds one pipeline stage so a bounded wait runs out."""
    lib().forge_debug_withhold_next_stage()
