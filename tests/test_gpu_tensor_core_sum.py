"""The GPU's weight gradient against the tensor-core accumulation model, bit for bit (needs a GB300).

The oracle's gradient is the exact sum over tokens rounded once to binary32; FORGE's exactness
statement (§2 Methodology, "Exactness") allows the fused kernel to differ from it only in how that
sum is ordered and rounded.  These tests show that the whole difference is the tensor core's
documented-by-measurement accumulation (tests/tensor_core_sum.py):
  * forge_dw_gemm's dW equals the model's sum exactly, for bf16 and E4M3 operands, on the
    workloads' layer shapes and token counts;
  * the fused step, at sampled elements, equals the oracle's update evaluated at the model's
    gradient with no allowance for the gradient's deviation;
  * over whole layers, the largest deviation of the GPU's dW from the exact sum is what the
    moment tolerance (compare.moment_rtol) is derived from.
"""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import fp8, step as ostep
from tests.compare import assert_moments, assert_weights, moment_rtol
from tests.helpers import bits, f32
from tests.tensor_core_sum import tc_dw_at
from workloads import (OPTIMIZERS, WORKLOADS, Layer, Workload, activations, activations_fp8, default_hparams,
                       layer_state, sample_positions)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def _wl(d_out, d_in, T):
    return Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")


def _columns(t, idx):
    """Columns `idx` of a device tensor, as a host array of bf16 bits (or uint8 codes), and the
    positions of the requested columns among them."""
    u, inv = np.unique(np.asarray(idx), return_inverse=True)
    sub = t[:, torch.from_numpy(u).to(t.device)].cpu()
    return (bits(sub) if sub.dtype == torch.bfloat16 else sub.numpy()), inv


@pytest.mark.parametrize("d_out, d_in, T", [(4096, 4096, 4096), (4096, 4096, 8192), (14336, 4096, 4096),
                                            (4096, 14336, 4096), (2048, 1280, 100)])
def test_dw_gemm_equals_the_tensor_core_model(d_out, d_in, T):
    """4096^2 at the Llama and coverage token counts, the Llama gate and down shapes, and a ragged
    token tail on CTA pairs: every sampled element bit for bit."""
    dy, x = activations(_wl(d_out, d_in, T), 0, 1, seed=T + d_out, device="cuda")
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm(dy, x, dW)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    rows, cols = (np.asarray(a) for a in sample_positions(d_out, d_in, 4096, 1))
    a, ri = _columns(dy, rows)
    b, ci = _columns(x, cols)
    model = tc_dw_at(a, b, ri, ci, k=16)
    got = dW[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    diff = np.flatnonzero(got.view(np.uint32) != model.view(np.uint32))
    assert diff.size == 0, f"{diff.size} of {rows.size} differ, e.g. gpu {got[diff[:4]]} model {model[diff[:4]]}"


@pytest.mark.parametrize("T", [4096, 8192])
def test_dw_gemm_e4m3_equals_the_tensor_core_model(T):
    """E4M3 operands (32 products per MMA), per-tensor scales: dW = RN(sum * RN(s_dY s_X))."""
    d_out = d_in = 4096
    dyq, s_dy, xq, s_x = activations_fp8(_wl(d_out, d_in, T), 0, 1, seed=5, device="cuda")
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm_e4m3(dyq, xq, s_dy, s_x, dW)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    rows, cols = (np.asarray(a) for a in sample_positions(d_out, d_in, 4096, 2))
    a, ri = _columns(dyq, rows)
    b, ci = _columns(xq, cols)
    acc = tc_dw_at(a, b, ri, ci, k=32, decode=fp8.decode_e4m3)
    model = (acc * np.float32(np.float32(s_dy) * np.float32(s_x))).astype(np.float32)
    got = dW[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    assert np.array_equal(got.view(np.uint32), model.view(np.uint32))


@pytest.mark.parametrize("opt", OPTIMIZERS)
def test_fused_step_equals_the_oracle_at_the_hardware_gradient(opt):
    """CTA pairs, T = 4096, sampled elements: with the tensor core's gradient in place of the exact
    one, the oracle's step and the fused kernel agree to the epilogue's own binary32 rounding
    (weights within one bf16 ULP, >= 99.9 % bit-identical, moments within 1e-6 relative), with no
    allowance for the gradient's summation deviation."""
    d_out, d_in, T = 2048, 1280, 4096
    wl = _wl(d_out, d_in, T)
    hp = default_hparams(opt, lr=1e-3)
    dy, x = activations(wl, 0, 1, seed=31, device="cuda")
    W, M, V = layer_state(wl, 0, opt, seed=32, device="cuda")
    rows, cols = (np.asarray(a) for a in sample_positions(d_out, d_in, 4096, 3))
    ri_t, ci_t = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    w0 = bits(W[ri_t, ci_t])
    m0 = None if M is None else f32(M[ri_t, ci_t])
    v0 = None if V is None else f32(V[ri_t, ci_t])
    fg.fused_dw_step(dy, x, W, M, V, None, opt, hp, 4, seed=7)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    a, ri = _columns(dy, rows)
    b, ci = _columns(x, cols)
    g = tc_dw_at(a, b, ri, ci, k=16)
    e = (rows * d_in + cols).astype(np.uint64)
    ref = ostep.apply_update(opt, g, w0, m0, v0, hp, 4, 7, e)
    assert_weights(bits(W[ri_t, ci_t]), ref["W"], "W", w_old_bits=w0)
    if M is not None:
        assert_moments(f32(M[ri_t, ci_t]), ref["m"], "m", rtol=1e-6)
    if V is not None:
        assert_moments(f32(V[ri_t, ci_t]), ref["v"], "v", rtol=1e-6)


@pytest.mark.parametrize("workload, layer", [("llama8b-mlp", 0), ("llama8b-mlp", 2), ("qwen14b-sweep", 0)])
def test_whole_layer_deviation_sets_the_moment_tolerance(workload, layer):
    """Every element of a full-size layer (Llama-3.1-8B gate and down at T = 4096, Qwen3-14B q at
    T = 8192): the GPU's dW against the exact sum (float64 products summed in float64 on the GPU,
    then rounded to binary32; checked against the oracle's own sum at sampled positions).  The
    largest deviation relative to max(|exact|, rms(exact)) stays within compare.moment_rtol(T), and
    that tolerance is at most 1.5 times the deviation measured here."""
    wl = WORKLOADS[workload]
    l = wl.layers[layer]
    dy, x = activations(wl, layer, 1, device="cuda")
    dW = torch.empty(l.d_out, l.d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm(dy, x, dW)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    exact = (dy.double().t() @ x.double()).float()
    rows, cols = (np.asarray(a) for a in sample_positions(l.d_out, l.d_in, 1024, 4))
    a, ri = _columns(dy, rows)
    b, ci = _columns(x, cols)
    ref = ostep.dw_at(a, b, ri, ci)
    ex_s = exact[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    assert np.array_equal(ex_s.view(np.uint32), ref.view(np.uint32)), "float64 GEMM reference is not exact"
    e64 = exact.double()
    scale = torch.maximum(e64.abs(), e64.square().mean().sqrt())
    dev = float(((dW.double() - e64).abs() / scale).max())
    rt = moment_rtol(wl.T)
    print(f"{workload} layer {layer} T={wl.T}: max deviation {dev:.3e}, tolerance {rt:.3e} ({rt / dev:.2f}x)")
    assert dev <= rt
    assert rt <= 1.5 * dev
