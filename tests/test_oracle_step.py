"""Pins for the oracle's whole step (CPU only)."""
import numpy as np
import pytest

from oracle import bf16, int8_block, optim, philox, step
from tests.helpers import bits, f32
from workloads import WORKLOADS, Hparams, activations, default_hparams, layer_state


def _tiny_inputs(opt="adamw", t=1):
    wl = WORKLOADS["tiny"]
    dy, x = activations(wl, 0, t)
    w, m, v = layer_state(wl, 0, opt)
    return bits(dy), bits(x), bits(w), (None if m is None else f32(m)), (None if v is None else f32(v))


def test_tile_schedule_equals_full_gradient_schedule():
    """The summary's exactness claim for element-wise optimizers: applying the update
    tile by tile (128 x 128) gives the same result as one update on the full gradient."""
    dy, x, w, m, v = _tiny_inputs()
    m = np.abs(np.random.default_rng(0).standard_normal(w.shape)).astype(np.float32) * 1e-4
    v = np.random.default_rng(1).random(w.shape).astype(np.float32) * 1e-6
    hp = Hparams(lr=1e-3, weight_decay=0.01)
    full = step.fused_step("adamw", dy, x, w, m, v, hp, 3, seed=9)
    d_out, d_in = w.shape
    W = np.empty_like(w)
    M = np.empty_like(m)
    V = np.empty_like(v)
    for r0 in range(0, d_out, 128):
        for c0 in range(0, d_in, 128):
            sl = (slice(r0, r0 + 128), slice(c0, c0 + 128))
            g_tile = step.dw(dy[:, sl[0]], x[:, sl[1]])
            e = (np.arange(r0, r0 + 128)[:, None] * d_in + np.arange(c0, c0 + 128)[None, :]).astype(np.uint64)
            out = step.apply_update("adamw", g_tile, w[sl], m[sl], v[sl], hp, 3, 9, e)
            W[sl], M[sl], V[sl] = out["W"], out["m"], out["v"]
    np.testing.assert_array_equal(W, full["W"])
    np.testing.assert_array_equal(M, full["m"])
    np.testing.assert_array_equal(V, full["v"])


def test_adamw_first_step_moves_each_weight_by_about_lr():
    """t = 1 from zero moments: |W' - W(1 - lr wd)| = lr |g|/(|g| + eps) ~ lr, up to bf16 rounding."""
    dy, x, w, m, v = _tiny_inputs()
    hp = Hparams(lr=1e-3, weight_decay=0.01)
    out = step.fused_step("adamw", dy, x, w, m, v, hp, 1, seed=0)
    w64 = bf16.to_f64(w)
    moved = out["w_f32"].astype(np.float64) - w64 * (1 - optim.binary32(1e-3) * optim.binary32(0.01))
    g = out["g"].astype(np.float64)
    expect = -optim.binary32(1e-3) * g / (np.abs(g) + optim.binary32(1e-8))
    np.testing.assert_allclose(moved, expect, rtol=0, atol=2 * np.spacing(np.abs(w64).max().astype(np.float32)))
    # the stored bf16 weight is one of the two neighbours of the binary32 result
    lo = bf16.to_f64(bf16.round_nearest_even(out["w_f32"]))
    assert np.all(np.abs(bf16.to_f64(out["W"]) - out["w_f32"]) <= bf16.ulp(bf16.round_nearest_even(out["w_f32"])) + 1e-30)
    assert lo.shape == out["W"].shape


@pytest.mark.parametrize("opt", optim.OPTIMIZERS)
def test_sampled_step_equals_dense_step(opt):
    dy, x, w, m, v = _tiny_inputs(opt, t=2)
    hp = default_hparams(opt, lr=1e-3)
    dense = step.fused_step(opt, dy, x, w, m, v, hp, 2, seed=5)
    rows = np.array([0, 1, 100, 511, 300])
    cols = np.array([0, 255, 17, 128, 64])
    smp = step.fused_step_at(opt, dy, x, w, m, v, hp, 2, 5, rows, cols)
    np.testing.assert_array_equal(smp["W"], dense["W"][rows, cols])
    for k in ("m", "v"):
        if dense[k] is not None:
            np.testing.assert_array_equal(smp[k], dense[k][rows, cols])


def test_int8_blocks_equal_dense_int8_step():
    dy, x, w, _, _ = _tiny_inputs()
    rng = np.random.default_rng(4)
    m32 = (rng.standard_normal(w.shape) * 1e-4).astype(np.float32)
    v32 = (rng.random(w.shape) * 1e-6).astype(np.float32)
    mq, ms = int8_block.quantize(m32)
    vq, vs = int8_block.quantize(v32)
    hp = Hparams(lr=1e-3)
    dense = step.fused_step("adamw", dy, x, w, mq, vq, hp, 4, 1, "int8", ms, vs)
    rows = np.array([3, 3, 400])
    col0 = np.array([0, 192, 64])
    blk = step.fused_step_blocks("adamw", dy, x, w, mq, vq, hp, 4, 1, rows, col0, ms, vs)
    for b, (r, c) in enumerate(zip(rows, col0)):
        np.testing.assert_array_equal(blk["W"][b], dense["W"][r, c:c + 64])
        np.testing.assert_array_equal(blk["m"][b], dense["m"][r, c:c + 64])
        np.testing.assert_array_equal(blk["v"][b], dense["v"][r, c:c + 64])
        assert blk["m_scales"][b, 0] == dense["m_scales"][r, c // 64]
        assert blk["v_scales"][b, 0] == dense["v_scales"][r, c // 64]


def test_int8_update_uses_unquantised_new_moments():
    """The weight update of an INT8-state step equals the FP32-state step on the dequantised inputs."""
    dy, x, w, _, _ = _tiny_inputs()
    rng = np.random.default_rng(5)
    mq, ms = int8_block.quantize((rng.standard_normal(w.shape) * 1e-4).astype(np.float32))
    vq, vs = int8_block.quantize((rng.random(w.shape) * 1e-6).astype(np.float32))
    hp = Hparams(lr=1e-3)
    q = step.fused_step("adamw", dy, x, w, mq, vq, hp, 2, 3, "int8", ms, vs)
    f = step.fused_step("adamw", dy, x, w, int8_block.dequantize(mq, ms), int8_block.dequantize(vq, vs), hp, 2, 3)
    np.testing.assert_array_equal(q["W"], f["W"])
    np.testing.assert_array_equal(q["m_f32"], f["m"])


def test_sr_bits_follow_element_index_not_visit_order():
    e = np.arange(256, dtype=np.uint64)
    perm = np.random.default_rng(6).permutation(256)
    np.testing.assert_array_equal(philox.sr_bits(3, 4, e)[perm], philox.sr_bits(3, 4, e[perm]))


def test_sub_ulp_updates_accumulate_without_bias():
    """A fixed sub-ULP AdamW step, repeated, drifts the SR weights like the FP32 master (3 sigma)."""
    rng = np.random.default_rng(7)
    n = 4096
    w = bf16.round_nearest_even((rng.standard_normal(n) * 0.02).astype(np.float32))
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    hp = Hparams(lr=1e-6, weight_decay=0.0)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    master = bf16.to_f64(w)
    ws = w.copy()
    e = np.arange(n, dtype=np.uint64)
    steps = 200
    p_sum = np.zeros(n)
    for t in range(1, steps + 1):
        out = step.apply_update("adamw", g, ws, m, v, hp, t, 11, e)
        mm, vv = m.astype(np.float64), v.astype(np.float64)
        master, _, _ = optim.update("adamw", g.astype(np.float64), master, mm, vv, hp, t)
        frac = (out["w_f32"].astype(np.float64) - bf16.to_f64(bf16.stochastic_round(out["w_f32"], np.zeros(n, np.uint32))))
        p = np.abs(frac) / bf16.ulp(bf16.stochastic_round(out["w_f32"], np.zeros(n, np.uint32)))
        p_sum += p * (1 - p)
        ws, m, v = out["W"], out["m"], out["v"]
    u = bf16.ulp(w)
    diff = (bf16.to_f64(ws) - master) / u
    sigma = np.sqrt(p_sum.sum()) / n
    assert abs(diff.mean()) < 3 * sigma + 1e-3
    # and the drift is real: the weights moved in the direction of the master update
    assert np.mean((bf16.to_f64(ws) - bf16.to_f64(w)) * np.sign(master - bf16.to_f64(w))) > 0
