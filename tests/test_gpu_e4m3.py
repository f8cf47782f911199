"""FP8 (E4M3) operands with per-tensor scales, CUDA path vs oracle (needs a GB300).

The tensor core sums E4M3 code products (kind::f8f6f4, 128 tokens per pipeline stage) in FP32;
the epilogue multiplies the finished gradient tile by s_dY * s_X before the optimizer.  The cases
cover every tile shape (one CTA on 128 x 128 and 128 x 256, a CTA pair), a ragged token tail and ragged rows and columns, every optimizer and state format.
"""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import fp8, int8_block
from tests.compare import (assert_codes, assert_moments, assert_weights, gradient_sensitivity, moment_rtol)
from tests.helpers import bits, f32
from workloads import (OPTIMIZERS, WORKLOADS, Layer, Workload, activations_fp8, default_hparams, layer_state,
                       moment_init, sample_positions)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def _layer(d_out, d_in, T, opt, seed):
    wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
    dyq, s_dy, xq, s_x = activations_fp8(wl, 0, 1, seed)
    w, m, v = layer_state(wl, 0, opt, seed)
    return dyq, s_dy, xq, s_x, w, m, v


def _np8(t):
    return t.numpy().astype(np.uint8)


def _allow(opt, ref, w, m, v, hp, t, seed, T, state="fp32", ms=None, vs=None, what="w_f32"):
    """Per element, the movement of the oracle's binary32 output `what` under the gradient's
    allowed summation deviation (compare.gradient_sensitivity) for a whole layer."""
    e = np.arange(w.numel(), dtype=np.uint64).reshape(w.shape)
    return gradient_sensitivity(opt, ref["g"], bits(w), m, v, hp, t, seed, e, moment_rtol(T), state, ms, vs,
                                what=what)


# (d_out, d_in, T, tile): a pair (40 pair tiles); 128 x 256 (90 tiles); 128 x 128 with a token tail;
# ragged rows and columns on pairs (2128 and 1296 are multiples of 16, not of 128; 54 pair tiles)
CASES = [(2048, 1280, 256, (256, 256, 2)), (1152, 2560, 256, (128, 256, 1)), (384, 384, 192, (128, 128, 1)),
         (2128, 1296, 100, (256, 256, 2))]


@pytest.mark.parametrize("d_out, d_in, T, tile", CASES)
def test_dw_gemm_e4m3_matches_oracle(d_out, d_in, T, tile):
    got = fg.launch_shape(d_out, d_in, T)
    # the query answers for bf16 operands; E4M3 rows hold 128 elements, so where it says 128 x 64
    # E4M3 operands run on 128 x 128
    cols = 128 if got["tile_cols"] == 64 else got["tile_cols"]
    assert (got["tile_rows"], cols, got["cluster"]) == tile
    dyq, s_dy, xq, s_x, *_ = _layer(d_out, d_in, T, "sgd", seed=d_in + T)
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm_e4m3(dyq.cuda(), xq.cuda(), s_dy, s_x, dW)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    assert_moments(dW.cpu().numpy(), fp8.dw_fp8(_np8(dyq), _np8(xq), s_dy, s_x), "dW", rtol=moment_rtol(T))


def test_dw_gemm_e4m3_is_exact_on_integer_patterns():
    """Small integer codes, one nonzero per token column pattern: every sum is exact in FP32, so any
    index mix-up (transposed, shifted or swapped halves of a stage) shows bit for bit."""
    T, d_out, d_in = 256, 256, 384
    one_to_eight = np.array([0x38, 0x40, 0x44, 0x48, 0x4A, 0x4C, 0x4E, 0x50], np.uint8)  # 1 .. 8
    dy = np.zeros((T, d_out), np.uint8)
    x = np.zeros((T, d_in), np.uint8)
    dy[np.arange(d_out) % T, np.arange(d_out)] = one_to_eight[np.arange(d_out) % 7]
    x[(7 * np.arange(d_in)) % T, np.arange(d_in)] = one_to_eight[np.arange(d_in) % 5]
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm_e4m3(torch.from_numpy(dy).cuda(), torch.from_numpy(x).cuda(), 0.5, 0.25, dW)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dW.cpu().numpy(), fp8.dw_fp8(dy, x, 0.5, 0.25))


@pytest.mark.parametrize("opt", OPTIMIZERS)
@pytest.mark.parametrize("d_out, d_in", [(2048, 1280), (1152, 2560)])
def test_fused_e4m3_fp32_states(opt, d_out, d_in):
    T = 256
    dyq, s_dy, xq, s_x, w, m, v = _layer(d_out, d_in, T, opt, seed=3)
    hp = default_hparams(opt, lr=1e-3)
    dev = lambda t: None if t is None else t.cuda()
    W, M, V = dev(w), dev(m), dev(v)
    fg.fused_dw_step_e4m3(dyq.cuda(), xq.cuda(), s_dy, s_x, W, M, V, None, opt, hp, 4, seed=11)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    ref = fp8.fused_step_fp8(opt, _np8(dyq), _np8(xq), s_dy, s_x, bits(w), None if m is None else f32(m),
                             None if v is None else f32(v), hp, 4, 11)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w),
                   extra_tol=_allow(opt, ref, w, None if m is None else f32(m), None if v is None else f32(v), hp, 4,
                                    11, T))
    if m is not None:
        assert_moments(f32(M), ref["m"], "m")
    if v is not None:
        assert_moments(f32(V), ref["v"], "v")


def test_fused_e4m3_bf16_and_int8_states():
    T, d_out, d_in = 192, 2048, 1280
    dyq, s_dy, xq, s_x, w, m, v = _layer(d_out, d_in, T, "adamw", seed=4)
    hp = default_hparams("adamw", lr=1e-3)
    # BF16 states
    mb, vb = m.to(torch.bfloat16), v.to(torch.bfloat16)
    W, M, V = w.cuda(), mb.cuda(), vb.cuda()
    fg.fused_dw_step_e4m3(dyq.cuda(), xq.cuda(), s_dy, s_x, W, M, V, None, "adamw", hp, 2, seed=5)
    torch.cuda.synchronize()
    ref = fp8.fused_step_fp8("adamw", _np8(dyq), _np8(xq), s_dy, s_x, bits(w), bits(mb), bits(vb), hp, 2, 5,
                             state="bf16")
    allow = lambda what: _allow("adamw", ref, w, bits(mb), bits(vb), hp, 2, 5, T, "bf16", what=what)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=allow("w_f32"))
    assert_weights(bits(M), ref["m"], "m", w_old_bits=bits(mb), extra_tol=allow("m_f32"))
    assert_weights(bits(V), ref["v"], "v", w_old_bits=bits(vb), extra_tol=allow("v_f32"))
    # INT8 states
    rng = np.random.default_rng(4)
    m32 = (f32(moment_init("absnormal:1e-4", w.shape, 6)) * np.sign(rng.standard_normal(w.shape))).astype(np.float32)
    mq, ms = int8_block.quantize(m32)
    vq, vs = int8_block.quantize(f32(moment_init("uniform:1e-6", w.shape, 7)))
    W = w.cuda()
    M, V = torch.from_numpy(mq).cuda(), torch.from_numpy(vq).cuda()
    Q = torch.from_numpy(np.concatenate([ms.ravel(), vs.ravel()]).astype(np.float32)).cuda()
    fg.fused_dw_step_e4m3(dyq.cuda(), xq.cuda(), s_dy, s_x, W, M, V, Q, "adamw", hp, 3, seed=8)
    torch.cuda.synchronize()
    ref = fp8.fused_step_fp8("adamw", _np8(dyq), _np8(xq), s_dy, s_x, bits(w), mq, vq, hp, 3, 8, "int8", ms, vs)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w),
                   extra_tol=_allow("adamw", ref, w, mq, vq, hp, 3, 8, T, "int8", ms, vs))
    assert_codes(M.cpu().numpy(), ref["m"], "m codes")
    assert_codes(V.cpu().numpy(), ref["v"], "v codes")
    n64 = w.numel() // 64
    q = Q.cpu().numpy()
    assert_moments(q[:n64], ref["m_scales"].ravel(), "m scales")
    assert_moments(q[n64:], ref["v_scales"].ravel(), "v scales")


@pytest.mark.parametrize("d_out, d_in, T", [(2048, 1280, 320), (2128, 1296, 100), (512, 768, 320)])
def test_fused_e4m3_equals_unfused_bitwise(d_out, d_in, T):
    dyq, s_dy, xq, s_x, w, m, v = _layer(d_out, d_in, T, "adamw", seed=9)
    hp = default_hparams("adamw", lr=1e-3)
    D, X = dyq.cuda(), xq.cuda()
    W1, M1, V1 = w.cuda(), m.cuda(), v.cuda()
    W2, M2, V2 = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step_e4m3(D, X, s_dy, s_x, W1, M1, V1, None, "adamw", hp, 6, seed=1)
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm_e4m3(D, X, s_dy, s_x, dW)
    fg.opt_step(dW, W2, M2, V2, None, "adamw", hp, 6, seed=1)
    torch.cuda.synchronize()
    assert torch.equal(W1.view(torch.int16), W2.view(torch.int16))
    assert torch.equal(M1, M2) and torch.equal(V1, V2)


@pytest.mark.parametrize("opt", ["adamw", "lion"])
def test_e4m3_long_token_runs_on_pairs(opt):
    """T = 8192 on CTA pairs: 64 stages of 128 tokens per tile."""
    T, d_out, d_in = 8192, 2048, 1280
    assert fg.launch_shape(d_out, d_in, T)["cluster"] == 2
    dyq, s_dy, xq, s_x, w, m, v = _layer(d_out, d_in, T, opt, seed=10)
    hp = default_hparams(opt, lr=1e-3)
    W, M, V = w.cuda(), m.cuda(), None if v is None else v.cuda()
    fg.fused_dw_step_e4m3(dyq.cuda(), xq.cuda(), s_dy, s_x, W, M, V, None, opt, hp, 3, seed=2)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    ref = fp8.fused_step_fp8(opt, _np8(dyq), _np8(xq), s_dy, s_x, bits(w), f32(m), None if v is None else f32(v),
                             hp, 3, 2)
    rt = moment_rtol(T)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity(opt, ref["g"], bits(w), f32(m), None if v is None else f32(v), hp, 3, 2, e, rt)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    assert_moments(f32(M), ref["m"], "m", rtol=rt)


def test_llama8b_gate_e4m3_sampled():
    """Llama-3.1-8B MLP gate (14336 x 4096), T = 4096, E4M3 operands, AdamW with FP32 states."""
    wl = WORKLOADS["llama8b-mlp"]
    hp = default_hparams("adamw")
    dyq, s_dy, xq, s_x = activations_fp8(wl, 0, 1)
    w, m, v = layer_state(wl, 0, "adamw")
    W, M, V = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step_e4m3(dyq.cuda(), xq.cuda(), s_dy, s_x, W, M, V, None, "adamw", hp, 10, seed=4)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    d_out, d_in = w.shape
    rows, cols = (np.asarray(a) for a in sample_positions(d_out, d_in, 2048, 3))
    g = fp8.dw_fp8_at(_np8(dyq), _np8(xq), s_dy, s_x, rows, cols)
    from oracle import step as ostep
    e = (rows * d_in + cols).astype(np.uint64)
    ref = ostep.apply_update("adamw", g, bits(w)[rows, cols], f32(m)[rows, cols], f32(v)[rows, cols], hp, 10, 4, e)
    rt = moment_rtol(wl.T)
    extra = gradient_sensitivity("adamw", g, bits(w)[rows, cols], f32(m)[rows, cols], f32(v)[rows, cols], hp, 10, 4,
                                 e, rt)
    assert_weights(bits(W)[rows, cols], ref["W"], "W", w_old_bits=bits(w)[rows, cols], extra_tol=extra)
    assert_moments(f32(M)[rows, cols], ref["m"], "m", rtol=rt)
    assert_moments(f32(V)[rows, cols], ref["v"], "v", rtol=moment_rtol(wl.T, squared=True))


# ---------------------------------------------------------------------------- per-channel scales

def _layer_channels(d_out, d_in, T, opt, seed):
    """dY and X drawn as for the per-tensor cases, with columns of very different magnitudes, then
    quantised per column (workloads.fp8_e4m3_channels)."""
    from workloads import fp8_e4m3_channels
    g = torch.Generator().manual_seed(seed)
    dy = torch.randn(T, d_out, generator=g) * torch.logspace(-5, -2, d_out)[None, :]
    x = torch.randn(T, d_in, generator=g) * torch.logspace(-1, 1, d_in)[None, :]
    dyq, s_dy = fp8_e4m3_channels(dy)
    xq, s_x = fp8_e4m3_channels(x)
    wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
    w, m, v = layer_state(wl, 0, opt, seed)
    return dyq, s_dy, xq, s_x, w, m, v


@pytest.mark.parametrize("d_out, d_in, T", [(2048, 1280, 256), (1152, 2560, 256), (384, 384, 192),
                                            (2128, 1296, 100)])
def test_dw_gemm_e4m3_channel_scales(d_out, d_in, T):
    """Every tile shape; 1296 columns end 16 past a 32-column strip, so the last 4-column scale
    groups of a strip lie outside the layer."""
    dyq, s_dy, xq, s_x, *_ = _layer_channels(d_out, d_in, T, "sgd", seed=d_in + T)
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm_e4m3(dyq.cuda(), xq.cuda(), s_dy.cuda(), s_x.cuda(), dW)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    ref = fp8.dw_fp8(_np8(dyq), _np8(xq), s_dy.numpy(), s_x.numpy())
    assert_moments(dW.cpu().numpy(), ref, "dW", rtol=moment_rtol(T))


def test_constant_channel_scales_equal_the_tensor_scale_bitwise():
    dyq, s_dy, xq, s_x, w, m, v = _layer(2048, 1280, 256, "adamw", seed=12)
    hp = default_hparams("adamw", lr=1e-3)
    D, X = dyq.cuda(), xq.cuda()
    W1, M1, V1 = w.cuda(), m.cuda(), v.cuda()
    W2, M2, V2 = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step_e4m3(D, X, s_dy, s_x, W1, M1, V1, None, "adamw", hp, 3, seed=7)
    fg.fused_dw_step_e4m3(D, X, torch.full((2048,), s_dy, device="cuda"), torch.full((1280,), s_x, device="cuda"),
                          W2, M2, V2, None, "adamw", hp, 3, seed=7)
    torch.cuda.synchronize()
    assert torch.equal(W1.view(torch.int16), W2.view(torch.int16))
    assert torch.equal(M1, M2) and torch.equal(V1, V2)


@pytest.mark.parametrize("opt, state", [("adamw", "fp32"), ("lion", "fp32"), ("rmsprop", "fp32"), ("adamw", "bf16")])
def test_fused_e4m3_channel_scales(opt, state):
    T, d_out, d_in = 256, 2048, 1280
    dyq, s_dy, xq, s_x, w, m, v = _layer_channels(d_out, d_in, T, opt, seed=13)
    if state == "bf16":
        m, v = (None if t is None else t.to(torch.bfloat16) for t in (m, v))
    hp = default_hparams(opt, lr=1e-3)
    dev = lambda t: None if t is None else t.cuda()
    W, M, V = dev(w), dev(m), dev(v)
    fg.fused_dw_step_e4m3(dyq.cuda(), xq.cuda(), s_dy.cuda(), s_x.cuda(), W, M, V, None, opt, hp, 2, seed=9)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    mm = None if m is None else (bits(m) if state == "bf16" else f32(m))
    vv = None if v is None else (bits(v) if state == "bf16" else f32(v))
    ref = fp8.fused_step_fp8(opt, _np8(dyq), _np8(xq), s_dy.numpy(), s_x.numpy(), bits(w), mm, vv, hp, 2, 9,
                             state=state)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=_allow(opt, ref, w, mm, vv, hp, 2, 9, T, state))
    for got, old, key in ((M, m, "m"), (V, v, "v")):
        if got is None:
            continue
        if state == "bf16":
            assert_weights(bits(got), ref[key], key, w_old_bits=bits(old),
                           extra_tol=_allow(opt, ref, w, mm, vv, hp, 2, 9, T, state, what=key + "_f32"))
        else:
            assert_moments(f32(got), ref[key], key)


def test_fused_e4m3_channel_scales_equal_unfused_bitwise():
    dyq, s_dy, xq, s_x, w, m, v = _layer_channels(2128, 1296, 100, "adamw", seed=14)
    hp = default_hparams("adamw", lr=1e-3)
    D, X, SD, SX = dyq.cuda(), xq.cuda(), s_dy.cuda(), s_x.cuda()
    W1, M1, V1 = w.cuda(), m.cuda(), v.cuda()
    W2, M2, V2 = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step_e4m3(D, X, SD, SX, W1, M1, V1, None, "adamw", hp, 4, seed=3)
    dW = torch.empty(w.shape, dtype=torch.float32, device="cuda")
    fg.dw_gemm_e4m3(D, X, SD, SX, dW)
    fg.opt_step(dW, W2, M2, V2, None, "adamw", hp, 4, seed=3)
    torch.cuda.synchronize()
    assert torch.equal(W1.view(torch.int16), W2.view(torch.int16))
    assert torch.equal(M1, M2) and torch.equal(V1, V2)
