"""Ragged layers, CUDA path vs oracle (needs a GB300).

d_out and d_in need only be multiples of 8 (INT8 states: d_in a multiple of 64) and T is any
count: tiles that reach past the last row, column or token compute on TMA's zero fill, and the
epilogue skips device-memory accesses there.  Each case also checks that nothing outside the layer
is written: the tensors are views into larger buffers whose tails hold a guard pattern.
"""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import backward as obw, int8_block, step as ostep
from tests.compare import (assert_bf16_sum, assert_codes, assert_moments, assert_weights, gradient_sensitivity,
                           moment_rtol)
from tests.helpers import bits, f32
from workloads import Layer, Workload, activations, default_hparams, layer_state, moment_init

pytestmark = pytest.mark.gpu

GUARD = 4096  # extra elements after each buffer


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def _guarded(t):
    """A device copy of `t` at the start of a larger buffer whose tail is filled with a pattern."""
    flat = torch.empty(t.numel() + GUARD, dtype=t.dtype, device="cuda")
    flat[t.numel():] = _pattern(t.dtype)
    flat[:t.numel()] = t.reshape(-1).cuda()
    return flat, flat[:t.numel()].view(t.shape)


def _pattern(dtype):
    return {torch.bfloat16: 1.5, torch.float32: -7.25, torch.int8: 77}[dtype]


def _tail_intact(flat, n):
    tail = flat[n:].cpu()
    return bool((tail == _pattern(flat.dtype)).all())


def _layer(d_out, d_in, T, opt, seed):
    wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
    dy, x = activations(wl, 0, 1, seed)
    w, m, v = layer_state(wl, 0, opt, seed)
    return dy, x, w, m, v


# (d_out, d_in, T, tile): 128 x 64 with ragged rows, columns (d_in not a multiple of 16) and
# tokens; a CTA pair whose last row tile leaves one CTA wholly outside the layer (54 pair tiles);
# the same with 102 pair tiles, whose last 26 run as half tiles (the right half of the last tile
# column lies wholly past d_in); 128 x 256 with ragged columns (115 tiles); 128 x 128 with ragged
# rows and columns (110 tiles); an 8 x 8 layer with one token
CASES = [(200, 136, 100, (128, 64, 1)), (2056, 1288, 70, (256, 256, 2)), (4104, 1288, 70, (256, 256, 2)),
         (2944, 1032, 64, (128, 256, 1)), (1288, 1272, 90, (128, 128, 1)), (8, 8, 1, (128, 64, 1))]


@pytest.mark.parametrize("d_out, d_in, T, tile", CASES)
def test_launch_shape_of_ragged_layers(d_out, d_in, T, tile):
    got = fg.launch_shape(d_out, d_in, T)
    assert (got["tile_rows"], got["tile_cols"], got["cluster"]) == tile


@pytest.mark.parametrize("opt", ["adamw", "lion", "sgd", "rmsprop"])
@pytest.mark.parametrize("d_out, d_in, T, tile", CASES)
def test_fused_fp32_states_on_ragged_layers(opt, d_out, d_in, T, tile):
    dy, x, w, m, v = _layer(d_out, d_in, T, opt, seed=d_out + T)
    hp = default_hparams(opt, lr=1e-3)
    fw, W = _guarded(w)
    fm, M = _guarded(m) if m is not None else (None, None)
    fv, V = _guarded(v) if v is not None else (None, None)
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, opt, hp, 3, seed=17)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    ref = ostep.fused_step(opt, bits(dy), bits(x), bits(w), None if m is None else f32(m),
                           None if v is None else f32(v), hp, 3, 17)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity(opt, ref["g"], bits(w), None if m is None else f32(m),
                                 None if v is None else f32(v), hp, 3, 17, e, moment_rtol(T))
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    assert _tail_intact(fw, w.numel())
    for flat, got, old, key in ((fm, M, m, "m"), (fv, V, v, "v")):
        if old is not None:
            assert_moments(f32(got), ref[key], key)
            assert _tail_intact(flat, old.numel())


@pytest.mark.parametrize("d_out, d_in, T", [(200, 136, 100), (2056, 1288, 70), (4104, 1288, 70)])
def test_fused_bf16_states_on_ragged_layers(d_out, d_in, T):
    dy, x, w, m, v = _layer(d_out, d_in, T, "adamw", seed=5)
    m, v = m.to(torch.bfloat16), v.to(torch.bfloat16)
    hp = default_hparams("adamw", lr=1e-3)
    fw, W = _guarded(w)
    fm, M = _guarded(m)
    fv, V = _guarded(v)
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, "adamw", hp, 2, seed=6)
    torch.cuda.synchronize()
    ref = ostep.fused_step("adamw", bits(dy), bits(x), bits(w), bits(m), bits(v), hp, 2, 6, state="bf16")
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    args = ("adamw", ref["g"], bits(w), bits(m), bits(v), hp, 2, 6, e, moment_rtol(T), "bf16")
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=gradient_sensitivity(*args))
    assert_weights(bits(M), ref["m"], "m", w_old_bits=bits(m), extra_tol=gradient_sensitivity(*args, what="m_f32"))
    assert_weights(bits(V), ref["v"], "v", w_old_bits=bits(v), extra_tol=gradient_sensitivity(*args, what="v_f32"))
    for flat, t in ((fw, w), (fm, m), (fv, v)):
        assert _tail_intact(flat, t.numel())


@pytest.mark.parametrize("d_out, d_in, T", [(200, 320, 100), (2056, 1088, 70), (4104, 1088, 70)])
def test_fused_int8_states_on_ragged_layers(d_out, d_in, T):
    """d_in a multiple of 64 (1088 = 17 blocks, a ragged 256-column tile of a CTA pair), ragged rows
    and tokens; 4104 x 1088 has 85 pair tiles, whose last 9 run as half tiles (two warps per block;
    the right half of the last tile column lies wholly past d_in)."""
    dy, x, w, _, _ = _layer(d_out, d_in, T, "adamw", seed=7)
    rng = np.random.default_rng(7)
    m32 = (f32(moment_init("absnormal:1e-4", w.shape, 8)) * np.sign(rng.standard_normal(w.shape))).astype(np.float32)
    v32 = f32(moment_init("uniform:1e-6", w.shape, 9))
    mq, ms = int8_block.quantize(m32)
    vq, vs = int8_block.quantize(v32)
    hp = default_hparams("adamw", lr=1e-3)
    fw, W = _guarded(w)
    fm, M = _guarded(torch.from_numpy(mq))
    fv, V = _guarded(torch.from_numpy(vq))
    fq, Q = _guarded(torch.from_numpy(np.concatenate([ms.ravel(), vs.ravel()]).astype(np.float32)))
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, Q, "adamw", hp, 5, seed=12)
    torch.cuda.synchronize()
    ref = ostep.fused_step("adamw", bits(dy), bits(x), bits(w), mq, vq, hp, 5, 12, "int8", ms, vs)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity("adamw", ref["g"], bits(w), mq, vq, hp, 5, 12, e, moment_rtol(T), "int8", ms, vs)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    n64 = w.numel() // 64
    q = Q.cpu().numpy()
    assert_codes(M.cpu().numpy(), ref["m"], "m codes")
    assert_codes(V.cpu().numpy(), ref["v"], "v codes")
    assert_moments(q[:n64], ref["m_scales"].ravel(), "m scales")
    assert_moments(q[n64:], ref["v_scales"].ravel(), "v scales")
    for flat, n in ((fw, w.numel()), (fm, w.numel()), (fv, w.numel()), (fq, 2 * n64)):
        assert _tail_intact(flat, n)


@pytest.mark.parametrize("d_out, d_in, T", [(200, 136, 100), (2056, 1288, 70), (4104, 1288, 70)])
def test_fused_equals_unfused_on_ragged_layers(d_out, d_in, T):
    """The two-phase kernel's last warp is partly past the end (d_out d_in / 8 not a multiple of 32)."""
    dy, x, w, m, v = _layer(d_out, d_in, T, "adamw", seed=9)
    hp = default_hparams("adamw", lr=1e-3)
    D, X = dy.cuda(), x.cuda()
    W1, M1, V1 = w.cuda(), m.cuda(), v.cuda()
    fw, W2 = _guarded(w)
    fm, M2 = _guarded(m)
    fv, V2 = _guarded(v)
    fg.fused_dw_step(D, X, W1, M1, V1, None, "adamw", hp, 4, seed=2)
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm(D, X, dW)
    fg.opt_step(dW, W2, M2, V2, None, "adamw", hp, 4, seed=2)
    torch.cuda.synchronize()
    assert torch.equal(W1.view(torch.int16), W2.view(torch.int16))
    assert torch.equal(M1, M2) and torch.equal(V1, V2)
    for flat, t in ((fw, w), (fm, m), (fv, v)):
        assert _tail_intact(flat, t.numel())
    assert_moments(dW.cpu().numpy(), ostep.dw(bits(dy), bits(x)), "dW", rtol=moment_rtol(T))


@pytest.mark.parametrize("T, d_out, d_in", [(100, 200, 136), (70, 1096, 1288), (300, 8, 264), (4104, 520, 1288)])
def test_dx_on_ragged_layers(T, d_out, d_in):
    """dX with a ragged reduction (d_out), ragged columns (d_in not a multiple of 16: 16-byte stores);
    4104 tokens x 1288 columns make 102 pair tiles, whose last 26 run as half tiles."""
    dy = torch.randn(T, d_out, generator=torch.Generator().manual_seed(T)).mul(1e-3).to(torch.bfloat16)
    w = torch.randn(d_out, d_in, generator=torch.Generator().manual_seed(d_in)).mul(2e-2).to(torch.bfloat16)
    flat = torch.full((T * d_in + GUARD,), _pattern(torch.bfloat16), dtype=torch.bfloat16, device="cuda")
    dX = flat[:T * d_in].view(T, d_in)
    fg.dx_gemm(dy.cuda(), w.cuda(), dX)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    assert_bf16_sum(bits(dX), obw.dx_f32(bits(dy), bits(w)), d_out)
    assert _tail_intact(flat, T * d_in)
