"""CUDA path vs oracle, element by element, through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import int8_block, step as ostep
from tests.compare import assert_codes, assert_moments, assert_weights, gradient_sensitivity, moment_rtol
from tests.helpers import bits, f32
from tests.shapes import FEW_PAIRS, MID, PAIR, PAIR_MANY, SMALL, TILE, WIDE
from workloads import (OPTIMIZERS, WORKLOADS, Hparams, Layer, Workload, activations, default_hparams,
                       layer_state, moment_init, normal_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def dev(t):
    return None if t is None else t.cuda()


def _layer(d_out, d_in, T, opt, seed=0, dy_std=1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6"):
    wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, dy_std, m_init=m_init, v_init=v_init)
    dy, x = activations(wl, 0, 1, seed)
    w, m, v = layer_state(wl, 0, opt, seed)
    return dy, x, w, m, v


# ---------------------------------------------------------------------------- weight gradient

@pytest.mark.parametrize("d_out, d_in, T", [(128, 128, 64), (512, 256, 256), (384, 640, 192), PAIR + (320,),
                                            WIDE + (128,), PAIR_MANY + (128,)])
def test_dw_gemm_matches_oracle(d_out, d_in, T):
    dy = normal_bf16((T, d_out), 1e-2, seed=d_out + T)
    x = normal_bf16((T, d_in), 1.0, seed=d_in + 7 * T)
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm(dy.cuda(), x.cuda(), dW)
    torch.cuda.synchronize()
    ref = ostep.dw(bits(dy), bits(x))
    assert_moments(dW.cpu().numpy(), ref, "dW")


def test_dw_gemm_is_not_transposed_or_shifted():
    """Distinct integer patterns per (row, col): any index mix-up in the tile mapping shows."""
    T, d_out, d_in = 64, 256, 384
    dy = torch.zeros(T, d_out)
    x = torch.zeros(T, d_in)
    dy[torch.arange(d_out) % T, torch.arange(d_out)] = (torch.arange(d_out) % 7 + 1).float()
    x[torch.arange(d_in) % T, torch.arange(d_in)] = (torch.arange(d_in) % 5 + 1).float()
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm(dy.bfloat16().cuda(), x.bfloat16().cuda(), dW)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dW.cpu().numpy(), ostep.dw(bits(dy.bfloat16()), bits(x.bfloat16())))


# ---------------------------------------------------------------------------- optimizer epilogue alone

@pytest.mark.parametrize("opt", OPTIMIZERS)
def test_opt_step_matches_oracle_fp32(opt):
    dy, x, w, m, v = _layer(256, 384, 128, opt)
    g = ostep.dw(bits(dy), bits(x))
    hp = default_hparams(opt, lr=1e-3)
    t = 3
    W, M, V = dev(w), dev(m), dev(v)
    fg.opt_step(torch.from_numpy(g).cuda(), W, M, V, None, opt, hp, t, seed=77)
    torch.cuda.synchronize()
    e = np.arange(w.numel(), dtype=np.uint64).reshape(w.shape)
    ref = ostep.apply_update(opt, g, bits(w), None if m is None else f32(m), None if v is None else f32(v),
                             hp, t, 77, e)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w))
    if m is not None:
        assert_moments(f32(M), ref["m"], "m")
    if v is not None:
        assert_moments(f32(V), ref["v"], "v")


def _int8_state(shape, seed):
    m32 = f32(moment_init("absnormal:1e-4", shape, seed)) * np.sign(np.random.default_rng(seed).standard_normal(shape))
    v32 = f32(moment_init("uniform:1e-6", shape, seed + 1))
    mq, ms = int8_block.quantize(m32.astype(np.float32))
    vq, vs = int8_block.quantize(v32)
    return mq, ms, vq, vs


def _qscales_tensor(ms, vs):
    return torch.from_numpy(np.concatenate([ms.ravel(), vs.ravel()]).astype(np.float32)).cuda()


@pytest.mark.parametrize("opt", [o for o in OPTIMIZERS if o != "sgd"])
def test_opt_step_matches_oracle_int8(opt):
    dy, x, w, _, _ = _layer(256, 256, 128, opt)
    g = ostep.dw(bits(dy), bits(x))
    mq, ms, vq, vs = _int8_state(w.shape, 5)
    hp = default_hparams(opt, lr=1e-3)
    W = dev(w)
    M, V = torch.from_numpy(mq).cuda(), torch.from_numpy(vq).cuda()
    Q = _qscales_tensor(ms, vs)
    fg.opt_step(torch.from_numpy(g).cuda(), W, M, V, Q, opt, hp, 2, seed=3)
    torch.cuda.synchronize()
    e = np.arange(w.numel(), dtype=np.uint64).reshape(w.shape)
    ref = ostep.apply_update(opt, g, bits(w), mq, vq, hp, 2, 3, e, "int8", ms, vs)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w))
    q = Q.cpu().numpy()
    n64 = w.numel() // 64
    if ref["m"] is not None:
        assert_codes(M.cpu().numpy(), ref["m"], "m codes")
        assert_moments(q[:n64], ref["m_scales"].ravel(), "m scales")
    if ref["v"] is not None:
        assert_codes(V.cpu().numpy(), ref["v"], "v codes")
        assert_moments(q[n64:], ref["v_scales"].ravel(), "v scales")


# ---------------------------------------------------------------------------- the fused step

def test_tiny_workload_three_steps():
    """512 x 256 layer, T = 256, AdamW lr 1e-3, fresh X/dY each step, seed 0, 3 steps."""
    wl = WORKLOADS["tiny"]
    hp = Hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    w, m, v = layer_state(wl, 0, "adamw")
    W, M, V = w.cuda(), m.cuda(), v.cuda()
    rw, rm, rv = bits(w), f32(m), f32(v)
    for t in wl.steps:
        dy, x = activations(wl, 0, t)
        fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, "adamw", hp, t, seed=0)
        ref = ostep.fused_step("adamw", bits(dy), bits(x), rw, rm, rv, hp, t, 0)
        torch.cuda.synchronize()
        assert_weights(bits(W), ref["W"], f"W step {t}", w_old_bits=rw)
        assert_moments(f32(M), ref["m"], f"m step {t}")
        assert_moments(f32(V), ref["v"], f"v step {t}")
        rw, rm, rv = bits(W), f32(M), f32(V)  # continue from the GPU's state: per-step parity


# every tile kernel: a CTA pair on 256 x 256, one CTA on 128 x 256, one CTA on 128 x 128 (a layer
# whose few pair tiles would leave most SMs idle), one CTA on 128 x 64 (small layers)
SHAPES = [PAIR, PAIR_MANY, WIDE, MID, SMALL, FEW_PAIRS]


@pytest.mark.parametrize("opt, d_out, d_in", [(o,) + PAIR for o in OPTIMIZERS] + [(o,) + WIDE for o in OPTIMIZERS]
                         + [(o,) + SMALL for o in OPTIMIZERS]
                         + [(o,) + s for o in ("adamw", "nadam", "sgd") for s in (MID, FEW_PAIRS)])
def test_fused_matches_oracle_every_optimizer(opt, d_out, d_in):
    got = fg.launch_shape(d_out, d_in, 192)
    assert (got["tile_rows"], got["tile_cols"], got["cluster"]) == TILE[(d_out, d_in)]
    dy, x, w, m, v = _layer(d_out, d_in, 192, opt, seed=2)
    hp = default_hparams(opt, lr=1e-3)
    W, M, V = dev(w), dev(m), dev(v)
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, opt, hp, 4, seed=11)
    torch.cuda.synchronize()
    ref = ostep.fused_step(opt, bits(dy), bits(x), bits(w), None if m is None else f32(m),
                           None if v is None else f32(v), hp, 4, 11)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity(opt, ref["g"], bits(w), None if m is None else f32(m),
                                 None if v is None else f32(v), hp, 4, 11, e, moment_rtol(192))
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    if m is not None:
        assert_moments(f32(M), ref["m"], "m")
    if v is not None:
        assert_moments(f32(V), ref["v"], "v")


@pytest.mark.parametrize("opt, d_out, d_in", [(o, 256, 384) for o in OPTIMIZERS if o != "sgd"]
                         + [(o,) + PAIR for o in OPTIMIZERS if o != "sgd"] + [("adamw",) + WIDE, ("lion", 256, 768)]
                         + [(o,) + PAIR_MANY for o in ("adamw", "lion", "adagrad")])
def test_fused_int8_matches_oracle(opt, d_out, d_in):
    dy, x, w, _, _ = _layer(d_out, d_in, 128, opt, seed=4)
    mq, ms, vq, vs = _int8_state(w.shape, 9)
    hp = default_hparams(opt, lr=1e-3)
    W, M, V, Q = dev(w), torch.from_numpy(mq).cuda(), torch.from_numpy(vq).cuda(), _qscales_tensor(ms, vs)
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, Q, opt, hp, 5, seed=12)
    torch.cuda.synchronize()
    ref = ostep.fused_step(opt, bits(dy), bits(x), bits(w), mq, vq, hp, 5, 12, "int8", ms, vs)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity(opt, ref["g"], bits(w), mq, vq, hp, 5, 12, e, moment_rtol(128), "int8", ms, vs)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    q = Q.cpu().numpy()
    n64 = w.numel() // 64
    if ref["m"] is not None:
        assert_codes(M.cpu().numpy(), ref["m"], "m codes")
        assert_moments(q[:n64], ref["m_scales"].ravel(), "m scales")
    if ref["v"] is not None:
        assert_codes(V.cpu().numpy(), ref["v"], "v codes")
        assert_moments(q[n64:], ref["v_scales"].ravel(), "v scales")


@pytest.mark.parametrize("opt, T, shape", [("adamw", 8192, PAIR), ("lion", 6144, PAIR), ("rmsprop", 4096, PAIR),
                                          ("sgd_momentum", 8192, PAIR_MANY)])
def test_fused_int8_long_token_runs_match_oracle(opt, T, shape):
    """INT8 states on CTA pairs over long token runs (16 epilogue warps, rows staged in two
    halves, 5 operand stages); 4096 x 1280 ends on half tiles, where two warps share each block.
    Codes and scales against the oracle with the summation allowance of T tokens."""
    d_out, d_in = shape
    assert fg.launch_shape(d_out, d_in, T)["cluster"] == 2
    dy, x, w, _, _ = _layer(d_out, d_in, T, opt, seed=44)
    mq, ms, vq, vs = _int8_state(w.shape, 19)
    hp = default_hparams(opt, lr=1e-3)
    W, M, V, Q = dev(w), torch.from_numpy(mq).cuda(), torch.from_numpy(vq).cuda(), _qscales_tensor(ms, vs)
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, Q, opt, hp, 6, seed=23)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    ref = ostep.fused_step(opt, bits(dy), bits(x), bits(w), mq, vq, hp, 6, 23, "int8", ms, vs)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    rt = moment_rtol(T)
    extra = gradient_sensitivity(opt, ref["g"], bits(w), mq, vq, hp, 6, 23, e, rt, "int8", ms, vs)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    q = Q.cpu().numpy()
    n64 = w.numel() // 64
    if ref["m"] is not None:
        assert_codes(M.cpu().numpy(), ref["m"], "m codes")
        assert_moments(q[:n64], ref["m_scales"].ravel(), "m scales", rtol=rt)
    if ref["v"] is not None:
        assert_codes(V.cpu().numpy(), ref["v"], "v codes")
        assert_moments(q[n64:], ref["v_scales"].ravel(), "v scales", rtol=moment_rtol(T, squared=True))


@pytest.mark.parametrize("opt, d_out, d_in", [(o, d_out, d_in) for o in ("adamw", "lion", "adagrad")
                                               for d_out, d_in in SHAPES])
def test_fused_equals_unfused_bitwise(opt, d_out, d_in):
    """The summary's exactness statement on the GPU: same mainloop order, so the fused step and
    the two-phase step (dW to memory, then the optimizer) give identical bits."""
    dy, x, w, m, v = _layer(d_out, d_in, 256, opt, seed=6)
    hp = default_hparams(opt, lr=1e-3)
    W1, M1, V1 = dev(w), dev(m), dev(v)
    W2, M2, V2 = dev(w), dev(m), dev(v)
    D, X = dy.cuda(), x.cuda()
    fg.fused_dw_step(D, X, W1, M1, V1, None, opt, hp, 2, seed=5)
    dW = torch.empty(w.shape, dtype=torch.float32, device="cuda")
    fg.dw_gemm(D, X, dW)
    fg.opt_step(dW, W2, M2, V2, None, opt, hp, 2, seed=5)
    torch.cuda.synchronize()
    assert torch.equal(W1.view(torch.int16), W2.view(torch.int16))
    if m is not None:
        assert torch.equal(M1, M2)
    if v is not None:
        assert torch.equal(V1, V2)


@pytest.mark.parametrize("opt, d_out, d_in", [("adamw",) + PAIR, ("lion",) + WIDE, ("adagrad",) + PAIR_MANY])
def test_long_token_runs(opt, d_out, d_in):
    """T = 8192 (the coverage and Qwen3-14B workloads' token count) on CTA pairs and on 128 x 256
    tiles; 4096 x 1280 has 80 pair tiles, more than the 76 resident pairs, and runs its last 4 as
    half tiles."""
    T = 8192
    got = fg.launch_shape(d_out, d_in, T)
    assert (got["tile_rows"], got["tile_cols"], got["cluster"]) == TILE[(d_out, d_in)]
    dy, x, w, m, v = _layer(d_out, d_in, T, opt, seed=13)
    hp = default_hparams(opt, lr=1e-3)
    W, M, V = dev(w), dev(m), dev(v)
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, opt, hp, 3, seed=17)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    ref = ostep.fused_step(opt, bits(dy), bits(x), bits(w), None if m is None else f32(m),
                           None if v is None else f32(v), hp, 3, 17)
    rt = moment_rtol(T)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity(opt, ref["g"], bits(w), None if m is None else f32(m),
                                 None if v is None else f32(v), hp, 3, 17, e, rt)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    if m is not None:
        assert_moments(f32(M), ref["m"], "m", rtol=rt)
    if v is not None:
        assert_moments(f32(V), ref["v"], "v", rtol=moment_rtol(T, squared=True))


@pytest.mark.parametrize("d_out, d_in", [(2048, 2560), (4096, 1280), (2176, 2560), (2048, 1408)])
def test_many_tiles_with_a_ragged_persistent_tail(d_out, d_in):
    """More tiles than resident pairs or CTAs, not a multiple of them: 80 pair tiles of 256 x 256
    (2048 x 2560 and 4096 x 1280); 170 tiles of 128 x 256 (d_out not a multiple of 256); 176 tiles
    of 128 x 128."""
    dy, x, w, m, v = _layer(d_out, d_in, 128, "adamw", seed=8)
    hp = default_hparams("adamw", lr=1e-3)
    W, M, V = dev(w), dev(m), dev(v)
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, "adamw", hp, 7, seed=21)
    torch.cuda.synchronize()
    ref = ostep.fused_step("adamw", bits(dy), bits(x), bits(w), f32(m), f32(v), hp, 7, 21)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity("adamw", ref["g"], bits(w), f32(m), f32(v), hp, 7, 21, e, moment_rtol(128))
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    assert_moments(f32(M), ref["m"], "m")
    assert_moments(f32(V), ref["v"], "v")


def test_zero_tokens_is_a_zero_gradient_step():
    _, _, w, m, v = _layer(256, 128, 64, "adamw")
    hp = default_hparams("adamw", lr=1e-3)
    W, M, V = dev(w), dev(m), dev(v)
    empty = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    fg.fused_dw_step(empty, torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"), W, M, V, None, "adamw", hp,
                     3, seed=1)
    torch.cuda.synchronize()
    e = np.arange(w.numel(), dtype=np.uint64).reshape(w.shape)
    ref = ostep.apply_update("adamw", np.zeros(w.shape, np.float32), bits(w), f32(m), f32(v), hp, 3, 1, e)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w))
    assert_moments(f32(M), ref["m"])
    assert_moments(f32(V), ref["v"])


def test_empty_layer_is_a_no_op():
    z = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    fg.fused_dw_step(torch.empty(64, 0, dtype=torch.bfloat16, device="cuda"),
                     torch.empty(64, 128, dtype=torch.bfloat16, device="cuda"), z,
                     torch.empty(0, 128, device="cuda"), torch.empty(0, 128, device="cuda"), None, "adamw",
                     Hparams(), 1)
    assert fg.sync_status() == 0


def test_status_word_clean_after_normal_runs():
    assert fg.sync_status() == 0


@pytest.mark.parametrize("d_out, d_in, T, rows, cols, cluster", [
    (2048, 1280, 8192, 256, 256, 2), (2048, 1280, 64, 256, 256, 2), (1536, 1792, 64, 256, 256, 2),
    (1536, 1536, 64, 128, 128, 1), (1152, 2560, 64, 128, 256, 1), (1152, 2048, 64, 128, 128, 1),
    (384, 384, 64, 128, 64, 1), (512, 256, 256, 128, 64, 1), (1024, 1024, 4096, 128, 64, 1),
    (1280, 1280, 64, 128, 128, 1)])
def test_launch_shape_query(d_out, d_in, T, rows, cols, cluster):
    """Pairs once they fill more than half the SMs (1536 x 1792: 42 pair tiles; 1536 x 1536: 36, so
    144 tiles of 128 x 128); 128 x 256 likewise (1152 x 2560: 90 CTAs; 1152 x 2048: 72); 128 x 64
    once 128 x 128 would fill at most half (1024^2: 64 CTAs of 128 x 128, so 128 of 128 x 64;
    1280^2: 100 of 128 x 128)."""
    import ctypes
    shape = fg.ForgeShape(T=T, d_out=d_out, d_in=d_in, state=0, reserved=0)
    r, c, cl, n = (ctypes.c_int32() for _ in range(4))
    assert fg.lib().forge_launch_shape(ctypes.byref(shape), ctypes.byref(r), ctypes.byref(c), ctypes.byref(cl),
                                       ctypes.byref(n)) == 0
    assert (r.value, c.value, cl.value) == (rows, cols, cluster)
    tiles = (d_out // rows) * (d_in // cols)
    assert n.value == min(tiles * cluster, 152)  # one CTA per SM at most, one pair per pair tile
