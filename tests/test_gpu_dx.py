"""The input gradient dX = dY W and the layer backward, CUDA path vs oracle (needs a GB300).

dX runs on the same tile pipeline as the weight gradient with tokens as tile rows, so the cases
cover each tile shape (one CTA on 128 x 128 or 128 x 256, a CTA pair), a ragged token tail, more tiles than resident CTAs, and the layer backward's ordering: dX must come
from the weights before the fused step replaces them.
"""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import backward as obw, step as ostep
from tests.compare import (assert_bf16_sum, assert_moments, assert_weights, gradient_sensitivity,
                           moment_rtol)
from tests.helpers import bits, f32
from workloads import WORKLOADS, activations, default_hparams, layer_state, normal_bf16, sample_positions

pytestmark = pytest.mark.gpu

GUARD = 0x7FBF  # a NaN pattern the kernel never writes; rows past T must keep it


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def _inputs(T, d_out, d_in, seed):
    dy = normal_bf16((T, d_out), 1e-3, seed=seed)
    w = normal_bf16((d_out, d_in), 2e-2, seed=seed + 1)
    return dy, w


def _run_dx(dy, w, guard_rows=64):
    """dX into the first T rows of a buffer whose extra rows hold GUARD."""
    T, d_in = dy.shape[0], w.shape[1]
    buf = torch.full((T + guard_rows, d_in), GUARD, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fg.dx_gemm(dy.cuda(), w.cuda(), buf[:T])
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    out = buf.cpu()
    assert (bits(out[T:]) == GUARD).all(), "dX wrote past the last token row"
    return out[:T]


# (T, d_out, d_in) -> tile (a shape is taken only when it fills more than half the SMs): 128 x 64
# with a 64-token tail; 128 x 256 with T not a multiple of 256 (80 tiles); a CTA pair with a 64-token
# tail (90 pair tiles); a CTA pair, 170 tiles (more than resident pairs); a CTA pair on a long
# reduction (d_out = 8192, 40 pair tiles); few pair tiles and 128 x 128 tiles, so 128 x 64; 128 x
# 128 (90 tiles)
CASES = [(320, 256, 384, (128, 64, 1)), (640, 384, 4096, (128, 256, 1)), (2112, 512, 2560, (256, 256, 2)),
         (4160, 512, 2560, (256, 256, 2)), (1024, 8192, 2560, (256, 256, 2)), (576, 512, 768, (128, 64, 1)),
         (1152, 512, 1280, (128, 128, 1))]


@pytest.mark.parametrize("T, d_out, d_in, shape", CASES)
def test_dx_matches_oracle(T, d_out, d_in, shape):
    got = fg.dx_launch_shape(T, d_out, d_in)
    assert (got["tile_rows"], got["tile_cols"], got["cluster"]) == shape
    dy, w = _inputs(T, d_out, d_in, seed=T + d_in)
    out = _run_dx(dy, w)
    assert_bf16_sum(bits(out), obw.dx_f32(bits(dy), bits(w)), d_out)


@pytest.mark.parametrize("T", [1, 63, 64, 129])
def test_dx_short_token_runs(T):
    """Fewer tokens than one tile: the rest of the tile is zero fill and is not stored."""
    dy, w = _inputs(T, 256, 512, seed=40 + T)
    out = _run_dx(dy, w)
    assert_bf16_sum(bits(out), obw.dx_f32(bits(dy), bits(w)), 256)


def test_dx_identity_and_permutation_are_exact():
    """W = I returns dY bit for bit; a permutation moves columns exactly (one product per output)."""
    T, d = 320, 512
    dy = normal_bf16((T, d), 1.0, seed=50)
    eye = torch.eye(d, dtype=torch.bfloat16)
    assert torch.equal(_run_dx(dy, eye).view(torch.int16), dy.view(torch.int16))
    perm = torch.randperm(d, generator=torch.Generator().manual_seed(51))
    p = torch.zeros(d, d, dtype=torch.bfloat16)
    p[torch.arange(d), perm] = 1.0
    out = _run_dx(dy, p)
    assert torch.equal(out[:, perm].view(torch.int16), dy.view(torch.int16))


def test_dx_empty_and_zero_reduction():
    """T = 0 or d_in = 0: nothing to write; d_out = 0: dX is zero."""
    dX = torch.full((64, 256), 1.0, dtype=torch.bfloat16, device="cuda")
    empty_dy = torch.empty(64, 0, dtype=torch.bfloat16, device="cuda")
    empty_w = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    fg.dx_gemm(empty_dy, empty_w, dX)
    torch.cuda.synchronize()
    assert (dX == 0).all()
    fg.dx_gemm(torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"),
               torch.ones(128, 256, dtype=torch.bfloat16, device="cuda"),
               torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"))
    assert fg.sync_status() == 0


def _backward_case(opt, T, d_out, d_in, seed):
    from workloads import Layer, Workload
    wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
    dy, x = activations(wl, 0, 1, seed)
    w, m, v = layer_state(wl, 0, opt, seed)
    return dy, x, w, m, v


@pytest.mark.parametrize("opt, T, d_out, d_in", [("adamw", 512, 512, 768), ("lion", 256, 384, 384),
                                                 ("sgd", 192, 256, 512), ("adamw", 1024, 2048, 2560)])
def test_linear_backward_reads_weights_before_the_step(opt, T, d_out, d_in):
    """dX equals dY W_old (not dY W_new) and the weight step equals a separate fused step bit for bit."""
    dy, x, w, m, v = _backward_case(opt, T, d_out, d_in, seed=60)
    hp = default_hparams(opt, lr=5e-2)  # a large step, so dY W_new is far from dY W_old
    D, X = dy.cuda(), x.cuda()
    W1, M1, V1 = w.cuda(), None if m is None else m.cuda(), None if v is None else v.cuda()
    dX = torch.empty(T, d_in, dtype=torch.bfloat16, device="cuda")
    fg.linear_backward(D, X, W1, M1, V1, None, dX, opt, hp, 4, seed=9)
    W2, M2, V2 = w.cuda(), None if m is None else m.cuda(), None if v is None else v.cuda()
    fg.fused_dw_step(D, X, W2, M2, V2, None, opt, hp, 4, seed=9)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    assert torch.equal(W1.view(torch.int16), W2.view(torch.int16))
    for a, b in ((M1, M2), (V1, V2)):
        if a is not None:
            assert torch.equal(a, b)
    assert_bf16_sum(bits(dX.cpu()), obw.dx_f32(bits(dy), bits(w)), d_out)
    stale = obw.dx(bits(dy), bits(W1.cpu()))
    assert (bits(dX.cpu()) != stale).mean() > 0.5, "dX looks computed from the updated weights"
    ref = ostep.fused_step(opt, bits(dy), bits(x), bits(w), None if m is None else f32(m),
                           None if v is None else f32(v), hp, 4, 9)
    rt = moment_rtol(T)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity(opt, ref["g"], bits(w), None if m is None else f32(m),
                                 None if v is None else f32(v), hp, 4, 9, e, rt)
    assert_weights(bits(W1.cpu()), ref["W"], w_old_bits=bits(w), extra_tol=extra)


@pytest.mark.parametrize("layer", [0, 2])
def test_llama8b_dx_sampled(layer):
    """Llama-3.1-8B MLP gate (dY 4096 x 14336, W 14336 x 4096) and down (dY 4096 x 4096, W 4096 x
    14336), both on CTA pairs, T = 4096: sampled dX elements vs d_out-term dot products."""
    wl = WORKLOADS["llama8b-mlp"]
    dy, _ = activations(wl, layer, 1)
    w, _, _ = layer_state(wl, layer, "adamw")
    T, (d_out, d_in) = dy.shape[0], w.shape
    dX = torch.empty(T, d_in, dtype=torch.bfloat16, device="cuda")
    fg.dx_gemm(dy.cuda(), w.cuda(), dX)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    rows, cols = sample_positions(T, d_in, 4096, 70 + layer)
    ref = obw.dx_at(bits(dy), bits(w), rows, cols)
    assert_bf16_sum(bits(dX.cpu())[rows, cols], ref["f32"], d_out)
