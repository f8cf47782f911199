"""The C-ABI library builds, loads, exports what include/forge.h declares, and rejects bad
arguments on the host before touching a device (CPU only: no kernel is launched)."""
import ctypes
import os
import re

import pytest

import backward_optimizer_gb300 as fg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    fg.build()
    return fg.lib()


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(forge_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("forge_fused_dw_step", "forge_dw_gemm", "forge_opt_step", "forge_sync_status",
              "forge_status_string"):
        assert n in names


@pytest.mark.parametrize("name", _declared_functions())
def test_every_declared_symbol_is_exported(L, name):
    assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(7):
        assert L.forge_status_string(code)
    assert b"unknown" in L.forge_status_string(99)


def _shape(T=256, d_out=512, d_in=256, state=0, reserved=0):
    return fg.ForgeShape(T=T, d_out=d_out, d_in=d_in, state=state, reserved=reserved)


A = 0x10000  # aligned fake addresses: every call below is rejected before any dereference


def _fused(L, shape, opt=0, step=1, W=A, m=A, v=A, q=None, dY=A, X=A, hp=True):
    hps = fg.hparams_struct() if hp else None
    return L.forge_fused_dw_step(dY, X, W, m, v, q, opt, ctypes.byref(hps) if hps else None,
                                 ctypes.byref(shape) if shape is not None else None, step, 0, None)


@pytest.mark.parametrize("kw, code", [
    (dict(shape=None), 1),
    (dict(shape=_shape(d_out=500)), 1),
    (dict(shape=_shape(d_in=204)), 1),               # d_out and d_in: multiples of 8
    (dict(shape=_shape(state=1, d_in=200), q=A), 1),  # INT8 blocks of 64 may not span rows
    (dict(shape=_shape(T=-64)), 1),
    (dict(shape=_shape(reserved=1)), 1),
    (dict(shape=_shape(state=5)), 1),
    (dict(shape=_shape(), opt=9), 1),
    (dict(shape=_shape(), step=0), 1),
    (dict(shape=_shape(), hp=False), 1),
    (dict(shape=_shape(), W=None), 1),
    (dict(shape=_shape(), m=None), 1),
    (dict(shape=_shape(), v=None), 1),
    (dict(shape=_shape(state=1), q=None), 1),
    (dict(shape=_shape(state=1), opt=6, q=A), 2),
    (dict(shape=_shape(state=2), opt=6), 2),
    (dict(shape=_shape(state=3)), 1),
    (dict(shape=_shape(), W=A + 8), 3),
    (dict(shape=_shape(), m=A + 16), 3),
    (dict(shape=_shape(), dY=A + 2), 3),
    (dict(shape=_shape(), X=None), 1),
])
def test_fused_rejects_bad_arguments_on_host(L, kw, code):
    shape = kw.pop("shape")
    assert _fused(L, shape, **kw) == code


def test_unused_moments_may_be_null(L):
    # SGD uses neither moment: only the device step can fail here (no GPU on a CPU machine)
    if _cuda_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    st = _fused(L, _shape(), opt=6, m=None, v=None)
    assert st == 4  # FORGE_ERR_CUDA: argument checks passed, no device


def test_dw_gemm_and_opt_step_reject_bad_arguments(L):
    assert L.forge_dw_gemm(A, A, None, ctypes.byref(_shape()), None) == 1
    assert L.forge_dw_gemm(A, A, A + 4, ctypes.byref(_shape()), None) == 3
    assert L.forge_dw_gemm(A, A, A, ctypes.byref(_shape(d_in=60)), None) == 1
    hp = fg.hparams_struct()
    assert L.forge_opt_step(A, None, A, A, None, 0, ctypes.byref(hp), ctypes.byref(_shape()), 1, 0, None) == 1
    assert L.forge_opt_step(A + 4, A, A, A, None, 0, ctypes.byref(hp), ctypes.byref(_shape()), 1, 0, None) == 3
    assert L.forge_opt_step(A, A, A, A, None, 0, ctypes.byref(hp), ctypes.byref(_shape()), 0, 0, None) == 1


def test_dx_gemm_rejects_bad_arguments(L):
    s = ctypes.byref(_shape(T=100))  # any token count is accepted for dX
    assert L.forge_dx_gemm(A, A, None, s, None) == 1
    assert L.forge_dx_gemm(A, A, A + 2, s, None) == 3
    assert L.forge_dx_gemm(None, A, A, s, None) == 1
    assert L.forge_dx_gemm(A, A + 16, A, s, None) == 3
    assert L.forge_dx_gemm(A, A, A, ctypes.byref(_shape(d_in=204)), None) == 1
    assert L.forge_dx_gemm(A, A, A, None, None) == 1
    # empty dX: nothing is checked beyond the shape and nothing runs
    assert L.forge_dx_gemm(None, None, None, ctypes.byref(_shape(T=0)), None) == 0
    assert L.forge_dx_gemm(None, None, None, ctypes.byref(_shape(d_in=0)), None) == 0


def _backward(L, shape, dX=A, **kw):
    hp = fg.hparams_struct()
    args = dict(dY=A, X=A, W=A, m=A, v=A, q=None, opt=0, step=1)
    args.update(kw)
    return L.forge_linear_backward(args["dY"], args["X"], args["W"], args["m"], args["v"], args["q"], dX,
                                   args["opt"], ctypes.byref(hp), ctypes.byref(shape), args["step"], 0, None)


def test_linear_backward_checks_both_calls_before_launching(L):
    assert _backward(L, _shape(), dX=None) == 1        # dX missing: nothing launched
    assert _backward(L, _shape(), dX=A + 8) == 3
    assert _backward(L, _shape(d_out=100)) == 1        # d_out a multiple of 8
    assert _backward(L, _shape(), step=0) == 1
    assert _backward(L, _shape(), m=None) == 1
    if not _cuda_available():
        assert _backward(L, _shape()) == 4             # arguments pass; no device here


def test_wait_limit_setter_and_launch_counter(L):
    L.forge_set_wait_limit_ns(5)
    L.forge_set_wait_limit_ns(2_000_000_000)
    assert L.forge_launch_count() >= 0


def _cuda_available():
    import torch
    return torch.cuda.is_available()


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(fg, "_lib", None)
    monkeypatch.setattr(fg, "_LIB_PATH", "/nonexistent/libforge.so")
    with pytest.raises(fg.ForgeUnavailable):
        fg.lib()


def test_e4m3_entry_points_reject_bad_arguments(L):
    hp = fg.hparams_struct()

    def fused(shape, sdy=1.0, sx=1.0, opt=0):
        return L.forge_fused_dw_step_e4m3(A, A, sdy, sx, A, A, A, None, opt, ctypes.byref(hp), ctypes.byref(shape),
                                          1, 0, None)
    assert fused(_shape(d_out=520)) == 1            # E4M3 rows must be multiples of 16 bytes
    assert fused(_shape(d_in=264)) == 1
    assert fused(_shape(), sdy=0.0) == 1            # scales finite and positive
    assert fused(_shape(), sx=float("inf")) == 1
    assert fused(_shape(), sdy=float("nan")) == 1
    assert fused(_shape(), opt=9) == 1
    assert L.forge_dw_gemm_e4m3(A, A, 1.0, -2.0, A, ctypes.byref(_shape()), None) == 1
    assert L.forge_dw_gemm_e4m3(A, A, 1.0, 1.0, A + 4, ctypes.byref(_shape()), None) == 3
    if not _cuda_available():
        assert fused(_shape()) == 4                 # arguments pass; no device here


def test_binding_rejects_wrong_dtypes_and_shapes_before_the_library():
    """The Python binding checks dtypes and shapes on the host (CPU tensors suffice: the checks
    come before any device pointer is taken)."""
    import torch
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32)
    dy, x, w, m, v = bf(64, 128), bf(64, 256), bf(128, 256), f32(128, 256), f32(128, 256)
    with pytest.raises(TypeError):
        fg.fused_dw_step(dy, x, f32(128, 256), m, v)             # W must be bf16
    with pytest.raises(ValueError):
        fg.fused_dw_step(dy, x, bf(128, 128), m, v)              # W shape must be d_out x d_in
    with pytest.raises(ValueError):
        fg.fused_dw_step(dy, bf(32, 256), w, m, v)               # X must have dY's token count
    with pytest.raises(TypeError):
        fg.fused_dw_step(dy, x, w, m, bf(128, 256))              # m and v share one state dtype
    with pytest.raises(ValueError):
        fg.fused_dw_step(dy, x, w, torch.zeros(128, 256, dtype=torch.int8),
                         torch.zeros(128, 256, dtype=torch.int8))  # INT8 states need qscales
    with pytest.raises(TypeError):
        fg.fused_dw_step_e4m3(dy, x, 1.0, 1.0, w, m, v)          # E4M3 operands are one byte
    with pytest.raises(ValueError):
        fg.dx_gemm(dy, w, bf(64, 128))                           # dX is T x d_in
    with pytest.raises(TypeError):
        fg.dw_gemm(dy, x, bf(128, 256))                          # dW is FP32
    with pytest.raises(TypeError):
        fg.opt_step(bf(128, 256), w, m, v)                       # a materialised dW is FP32


def test_e4m3_channel_scales_reject_bad_vectors(L):
    hp = fg.hparams_struct()

    def fused(sdy, sx, shape=None):
        shape = shape or _shape()
        return L.forge_fused_dw_step_e4m3_channels(A, A, sdy, sx, A, A, A, None, 0, ctypes.byref(hp),
                                                   ctypes.byref(shape), 1, 0, None)
    assert fused(None, A) == 1
    assert fused(A, None) == 1
    assert fused(A + 4, A) == 3                         # 16-byte aligned vectors
    assert fused(A, A, _shape(d_in=264)) == 1           # E4M3 rows: multiples of 16 bytes
    assert L.forge_dw_gemm_e4m3_channels(A, A, A, A + 8, A, ctypes.byref(_shape()), None) == 3
    if not _cuda_available():
        assert fused(A, A) == 4


def test_header_compiles_as_c_and_a_c_program_links(L, tmp_path):
    """A C11 program (tests/c/abi_host.c) built with gcc -Wall -Werror against include/forge.h and
    libforge.so makes host-side calls through the C ABI."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    exe = tmp_path / "abi_host"
    libdir = os.path.dirname(fg.library_path())
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_host.c"), "-L", libdir, "-lforge",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


def test_hyperparameter_struct_follows_a_mutable_object():
    """A schedule that changes the fields of its hyperparameter object between steps is seen on the
    next call; immutable objects (workloads.Hparams) are converted once and reused."""
    import backward_optimizer_gb300 as fg
    from workloads import Hparams

    class Schedule:
        lr = 1e-3
        weight_decay = 0.0
    hp = Schedule()
    assert fg._hp_arg(hp)._obj.lr == pytest.approx(1e-3)
    hp.lr = 5e-2
    assert fg._hp_arg(hp)._obj.lr == pytest.approx(5e-2)
    frozen = Hparams(lr=2e-3)
    assert fg._hp_arg(frozen)._obj is fg._hp_arg(Hparams(lr=2e-3))._obj
    assert fg._hp_arg({"lr": 3e-3})._obj.lr == pytest.approx(3e-3)


def test_layers_call_checks_every_layer_before_launching(L):
    """forge_fused_dw_step_layers: each layer is checked as forge_fused_dw_step would check it, and
    an error in any layer launches nothing (no device is needed to see the argument errors)."""
    hps = fg.hparams_struct()
    arr = (fg.ForgeLayer * 3)()
    for i in range(3):
        arr[i] = fg.ForgeLayer(0x10000, 0x10000, 0x10000, 0x10000, 0x10000, None, 256, 512, 256, i)
    call = lambda n, state=0, step=1: L.forge_fused_dw_step_layers(arr, n, state, 0, ctypes.byref(hps), step, None)
    assert call(0) == 0
    assert call(3, step=0) == 1                      # step < 1
    arr[2].W = 0x10008
    assert call(3) == 3                              # the third layer's W is misaligned
    assert call(2) == 4                              # the first two pass the checks; no device here
    arr[2].W = 0x10000
    arr[1].m = None
    assert call(3) == 1                              # AdamW keeps m
    arr[1].m = 0x10000
    assert call(3, state=1) == 1                     # INT8 states need qscales
    assert L.forge_fused_dw_step_layers(None, 2, 0, 0, ctypes.byref(hps), 1, None) == 1
