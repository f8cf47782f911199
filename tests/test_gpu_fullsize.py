"""Parity at the workloads' full sizes, in the launch configuration bench.py times (needs a GB300).

The oracle computes sampled outputs one by one (dW at a position is a T-term dot product;
the optimizer is element-wise), and properties that hold at any size are checked on every
element: the fused step equals the two-phase step bitwise, and sub-ULP updates accumulate
without bias under stochastic rounding.
"""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import bf16, int8_block, optim, step as ostep
from tests.compare import assert_codes, assert_moments, assert_weights, gradient_sensitivity, moment_rtol
from tests.helpers import bits, f32
from workloads import (OPTIMIZERS, WORKLOADS, Hparams, activations, default_hparams, layer_state,
                       sample_positions)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def _sampled_check(dy, x, w0, m0, v0, W, M, V, opt, hp, t, seed, n=2048, pos_seed=0):
    d_out, d_in = w0.shape
    rows, cols = sample_positions(d_out, d_in, n, pos_seed)
    rows, cols = np.asarray(rows), np.asarray(cols)
    ref = ostep.fused_step_at(opt, bits(dy), bits(x), bits(w0), None if m0 is None else f32(m0),
                              None if v0 is None else f32(v0), hp, t, seed, rows, cols)
    T = dy.shape[0]
    rt = moment_rtol(T)
    pick = lambda a: None if a is None else f32(a)[rows, cols]
    e = (rows * d_in + cols).astype(np.uint64)
    extra = gradient_sensitivity(opt, ref["g"], bits(w0)[rows, cols], pick(m0), pick(v0), hp, t, seed, e, rt)
    assert_weights(bits(W)[rows, cols], ref["W"], "W", w_old_bits=bits(w0)[rows, cols], extra_tol=extra)
    if m0 is not None:
        assert_moments(f32(M)[rows, cols], ref["m"], "m", rtol=moment_rtol(T))
    if v0 is not None:
        assert_moments(f32(V)[rows, cols], ref["v"], "v", rtol=moment_rtol(T, squared=True))


@pytest.mark.parametrize("layer", [0, 2])
def test_llama8b_mlp_layer_sampled(layer):
    """Llama-3.1-8B MLP gate (14336 x 4096) and down (4096 x 14336), T = 4096, AdamW at step 10."""
    wl = WORKLOADS["llama8b-mlp"]
    hp = default_hparams("adamw")
    dy, x = activations(wl, layer, 1)
    w, m, v = layer_state(wl, layer, "adamw")
    W, M, V = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, "adamw", hp, 10, seed=0x5EED + layer)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    _sampled_check(dy, x, w, m, v, W, M, V, "adamw", hp, 10, 0x5EED + layer, n=4096)


def test_llama8b_gate_fused_equals_two_phase_bitwise():
    """At full size the fused step and the two-phase step (dW to memory, then the optimizer)
    produce identical bits: the same tile mainloop accumulates dW in the same order."""
    wl = WORKLOADS["llama8b-mlp"]
    hp = default_hparams("adamw")
    dy, x = activations(wl, 0, 1)
    w, m, v = layer_state(wl, 0, "adamw")
    D, X = dy.cuda(), x.cuda()
    W1, M1, V1 = w.cuda(), m.cuda(), v.cuda()
    W2, M2, V2 = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step(D, X, W1, M1, V1, None, "adamw", hp, 10, seed=3)
    dW = torch.empty(w.shape, dtype=torch.float32, device="cuda")
    fg.dw_gemm(D, X, dW)
    fg.opt_step(dW, W2, M2, V2, None, "adamw", hp, 10, seed=3)
    torch.cuda.synchronize()
    assert torch.equal(W1.view(torch.int16), W2.view(torch.int16))
    assert torch.equal(M1, M2) and torch.equal(V1, V2)
    # and the gradient itself matches the oracle at sampled positions
    rows, cols = sample_positions(*w.shape, 2048, 5)
    ref = ostep.dw_at(bits(dy), bits(x), rows, cols)
    assert_moments(dW.cpu().numpy()[rows, cols], ref, "dW", rtol=moment_rtol(wl.T))


@pytest.mark.parametrize("opt", OPTIMIZERS)
def test_coverage_4096_five_steps(opt):
    """One 4096 x 4096 layer, T = 8192, fresh X/dY each step, 5 steps (RAdam: 10, to reach the
    rectified branch at t = 6), FP32 states, lr 1e-4, wd 0.01; parity checked at every step."""
    wl = WORKLOADS["coverage-4096"]
    hp = default_hparams(opt)
    w, m, v = layer_state(wl, 0, opt)
    W, M, V = w.cuda(), (None if m is None else m.cuda()), (None if v is None else v.cuda())
    steps = range(1, 11) if opt == "radam" else range(1, 6)
    for t in steps:
        dy, x = activations(wl, 0, t)
        w0, m0, v0 = W.cpu(), (None if M is None else M.cpu()), (None if V is None else V.cpu())
        fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, opt, hp, t, seed=7)
        torch.cuda.synchronize()
        _sampled_check(dy, x, w0, m0, v0, W, M, V, opt, hp, t, 7, n=1024, pos_seed=t)
    assert fg.sync_status() == 0


def test_int8_4096_sampled_blocks():
    """4096 x 4096, T = 2048, AdamW with INT8 block-64 moments: sampled whole blocks."""
    wl = WORKLOADS["int8-4096"]
    hp = default_hparams("adamw")
    dy, x = activations(wl, 0, 1)
    w, _, _ = layer_state(wl, 0, "adamw")
    rng = np.random.default_rng(0)
    mq, ms = int8_block.quantize((rng.standard_normal(w.shape) * 1e-4).astype(np.float32))
    vq, vs = int8_block.quantize((rng.random(w.shape) * 1e-6).astype(np.float32))
    W, M, V = w.cuda(), torch.from_numpy(mq).cuda(), torch.from_numpy(vq).cuda()
    Q = torch.from_numpy(np.concatenate([ms.ravel(), vs.ravel()])).cuda()
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, Q, "adamw", hp, 3, seed=9)
    torch.cuda.synchronize()
    rows, col0 = sample_positions(*w.shape, 512, 2, block=64)
    rows, col0 = np.asarray(rows), np.asarray(col0)
    ref = ostep.fused_step_blocks("adamw", bits(dy), bits(x), bits(w), mq, vq, hp, 3, 9, rows, col0, ms, vs)
    cols = col0[:, None] + np.arange(64)[None, :]
    assert_weights(bits(W)[rows[:, None], cols], ref["W"], "W", w_old_bits=bits(w)[rows[:, None], cols])
    assert_codes(M.cpu().numpy()[rows[:, None], cols], ref["m"], "m codes")
    assert_codes(V.cpu().numpy()[rows[:, None], cols], ref["v"], "v codes")
    q = Q.cpu().numpy()
    n64 = w.numel() // 64
    blk = rows * (w.shape[1] // 64) + col0 // 64
    assert_moments(q[blk], ref["m_scales"][:, 0], "m scales", rtol=moment_rtol(wl.T))
    assert_moments(q[n64 + blk], ref["v_scales"][:, 0], "v scales", rtol=moment_rtol(wl.T, squared=True))


def test_sub_ulp_updates_accumulate_without_bias():
    """1000 AdamW steps at lr = 1e-7 on fixed X/dY (4096 x 4096, T = 2048): each step moves a
    weight by ~1e-3 of a bfloat16 ULP.  Stochastic rounding must make the bf16 weights drift like
    the FP32-master oracle: the mean of (W_gpu - W_master) / ulp over sampled elements within
    3 sigma of 0 (sigma^2 = steps/6 per element, the variance of a uniformly placed SR draw), and
    the drift must follow the master's direction (round-to-nearest would leave W unchanged)."""
    wl = WORKLOADS["int8-4096"]
    hp = Hparams(lr=1e-7, weight_decay=0.0)
    steps = 1000
    dy, x = activations(wl, 0, 1)
    w, _, _ = layer_state(wl, 0, "adamw")
    W = w.cuda()
    M = torch.zeros(w.shape, dtype=torch.float32, device="cuda")
    V = torch.zeros(w.shape, dtype=torch.float32, device="cuda")
    D, X = dy.cuda(), x.cuda()
    for t in range(1, steps + 1):
        fg.fused_dw_step(D, X, W, M, V, None, "adamw", hp, t, seed=11)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    n = 1 << 15
    rows, cols = sample_positions(*w.shape, n, 3)
    rows, cols = np.asarray(rows), np.asarray(cols)
    g = ostep.dw_at(bits(dy), bits(x), rows, cols).astype(np.float64)
    master = bf16.to_f64(bits(w)[rows, cols])
    mm = np.zeros(n)
    vv = np.zeros(n)
    for t in range(1, steps + 1):
        master, mm, vv = optim.update("adamw", g, master, mm, vv, hp, t)
    w0 = bf16.to_f64(bits(w)[rows, cols])
    ulp = bf16.ulp(bits(w)[rows, cols])
    gpu = bf16.to_f64(bits(W)[rows, cols])
    diff = (gpu - master) / ulp
    sigma = np.sqrt(steps / 6.0) / np.sqrt(n)
    assert abs(diff.mean()) < 3 * sigma, (diff.mean(), sigma)
    moved = (gpu - w0) * np.sign(master - w0)
    assert moved.mean() > 0.5 * np.abs(master - w0).mean()


# ---------------------------------------------------------------------------- Qwen3-14B layer shapes

def _device_sampled_check(wl, layer, opt, t, seed, n=2048, pos_seed=0):
    """One fused step on a full-size layer whose inputs are drawn on the device; the oracle gets
    the sampled positions' inputs copied back (the dY and X columns they read, W/m/v there)."""
    l = wl.layers[layer]
    hp = default_hparams(opt)
    dev = torch.device("cuda")
    dy, x = activations(wl, layer, 1, device=dev)
    W, M, V = layer_state(wl, layer, opt, device=dev)
    rows, cols = (np.asarray(a) for a in sample_positions(l.d_out, l.d_in, n, pos_seed))
    ri_t, ci_t = torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)
    w0 = bits(W[ri_t, ci_t])
    m0 = None if M is None else f32(M[ri_t, ci_t])
    v0 = None if V is None else f32(V[ri_t, ci_t])
    ur, ri = np.unique(rows, return_inverse=True)
    uc, ci = np.unique(cols, return_inverse=True)
    dy_cols = bits(dy[:, torch.from_numpy(ur).to(dev)])
    x_cols = bits(x[:, torch.from_numpy(uc).to(dev)])
    fg.fused_dw_step(dy, x, W, M, V, None, opt, hp, t, seed=seed)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    g = ostep.dw_at(dy_cols, x_cols, ri, ci)
    e = (rows * l.d_in + cols).astype(np.uint64)
    ref = ostep.apply_update(opt, g, w0, m0, v0, hp, t, seed, e)
    rt = moment_rtol(wl.T)
    extra = gradient_sensitivity(opt, g, w0, m0, v0, hp, t, seed, e, rt)
    assert_weights(bits(W[ri_t, ci_t]), ref["W"], "W", w_old_bits=w0, extra_tol=extra)
    if M is not None:
        assert_moments(f32(M[ri_t, ci_t]), ref["m"], "m", rtol=rt)
    if V is not None:
        assert_moments(f32(V[ri_t, ci_t]), ref["v"], "v", rtol=moment_rtol(wl.T, squared=True))
    return fg.launch_shape(l.d_out, l.d_in, wl.T)


@pytest.mark.parametrize("layer, name", [(0, "q"), (1, "k"), (4, "gate"), (6, "down")])
def test_qwen14b_layer_sampled(layer, name):
    """Qwen3-14B-shaped layers at T = 8192 (q 5120 x 5120, k 1024 x 5120, gate 17408 x 5120, down
    5120 x 17408), AdamW with FP32 moments at step 10, sampled elements against the oracle.  Every
    shape runs on CTA pairs, most with more tiles than resident pairs."""
    wl = WORKLOADS["qwen14b-sweep"]
    assert wl.layers[layer].name.endswith(name)
    shape = _device_sampled_check(wl, layer, "adamw", 10, 0x5EED + layer, n=2048, pos_seed=layer)
    assert (shape["tile_rows"], shape["tile_cols"], shape["cluster"]) == (256, 256, 2)


def test_qwen14b_gate_fused_equals_two_phase_bitwise():
    """Every element of the largest Qwen3-14B layer (gate, 17408 x 5120, T = 8192): the fused step
    and the two-phase step agree bit for bit."""
    wl = WORKLOADS["qwen14b-sweep"]
    hp = default_hparams("adamw")
    dev = torch.device("cuda")
    dy, x = activations(wl, 4, 1, device=dev)
    W1, M1, V1 = layer_state(wl, 4, "adamw", device=dev)
    W2, M2, V2 = W1.clone(), M1.clone(), V1.clone()
    fg.fused_dw_step(dy, x, W1, M1, V1, None, "adamw", hp, 10, seed=5)
    dW = torch.empty(W1.shape, dtype=torch.float32, device=dev)
    fg.dw_gemm(dy, x, dW)
    fg.opt_step(dW, W2, M2, V2, None, "adamw", hp, 10, seed=5)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    assert torch.equal(W1.view(torch.int16), W2.view(torch.int16))
    assert torch.equal(M1, M2) and torch.equal(V1, V2)
