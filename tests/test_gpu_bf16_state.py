"""BF16 optimizer states with stochastic rounding, CUDA path vs oracle (needs a GB300).

The moments are read as bfloat16, updated in binary32 and stored by stochastic rounding with
their own Philox streams.  Both sides draw the same bits, so the stored moments and weights are
bit-identical except where the binary32 value before rounding differs across a rounding boundary.
"""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import step as ostep
from tests.compare import assert_weights, gradient_sensitivity, moment_rtol
from tests.helpers import bits
from workloads import (OPTIMIZERS, WORKLOADS, Layer, Workload, activations, default_hparams, layer_state,
                       sample_positions)

pytestmark = pytest.mark.gpu

STATE_OPTS = [o for o in OPTIMIZERS if o != "sgd"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def _bf16(t):
    return None if t is None else t.to(torch.bfloat16)


def _layer(d_out, d_in, T, opt, seed):
    wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
    dy, x = activations(wl, 0, 1, seed)
    w, m, v = layer_state(wl, 0, opt, seed)
    return dy, x, w, _bf16(m), _bf16(v)


def _bits(t):
    return None if t is None else bits(t)


def _check(opt, dy, x, w, m, v, W, M, V, hp, t, seed, e=None, ref=None):
    """Weight and both moments against the oracle, each with its gradient sensitivity."""
    T = dy.shape[0]
    d_out, d_in = w.shape
    if ref is None:
        ref = ostep.fused_step(opt, bits(dy), bits(x), bits(w), _bits(m), _bits(v), hp, t, seed, state="bf16")
    if e is None:
        e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    rt = moment_rtol(T)
    args = (opt, ref["g"], bits(w), _bits(m), _bits(v), hp, t, seed, e, rt, "bf16")
    fracs = {"W": assert_weights(bits(W), ref["W"], "W", w_old_bits=bits(w),
                                 extra_tol=gradient_sensitivity(*args, what="w_f32"))}
    for name, old, new in (("m", m, M), ("v", v, V)):
        if old is not None:
            fracs[name] = assert_weights(bits(new), ref[name], name, w_old_bits=bits(old),
                                         extra_tol=gradient_sensitivity(*args, what=name + "_f32"))
    return fracs


@pytest.mark.parametrize("opt, d_out, d_in", [(o, 2048, 1280) for o in STATE_OPTS] + [(o, 1152, 2560) for o in STATE_OPTS]
                         + [(o, 384, 256) for o in ("adamw", "lion")])
def test_fused_bf16_states_match_oracle(opt, d_out, d_in):
    """512 x 512: a CTA pair; 384 x 256: one CTA on 128 x 256.  T = 256, step 3."""
    dy, x, w, m, v = _layer(d_out, d_in, 256, opt, seed=21)
    hp = default_hparams(opt, lr=1e-3)
    W, M, V = w.cuda(), None if m is None else m.cuda(), None if v is None else v.cuda()
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, opt, hp, 3, seed=31)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    _check(opt, dy, x, w, m, v, W.cpu(), None if M is None else M.cpu(), None if V is None else V.cpu(), hp, 3, 31)


@pytest.mark.parametrize("opt", ["adamw", "lion", "adagrad", "sgd_momentum"])
def test_fused_bf16_equals_unfused_bitwise(opt):
    """Fused step and two-phase step (dW to memory, then the optimizer kernel) agree bit for bit."""
    dy, x, w, m, v = _layer(2048, 1280, 320, opt, seed=22)
    hp = default_hparams(opt, lr=1e-3)
    dev = lambda t: None if t is None else t.cuda()
    D, X = dy.cuda(), x.cuda()
    W1, M1, V1 = dev(w), dev(m), dev(v)
    W2, M2, V2 = dev(w), dev(m), dev(v)
    fg.fused_dw_step(D, X, W1, M1, V1, None, opt, hp, 5, seed=3)
    dW = torch.empty(w.shape, dtype=torch.float32, device="cuda")
    fg.dw_gemm(D, X, dW)
    fg.opt_step(dW, W2, M2, V2, None, opt, hp, 5, seed=3)
    torch.cuda.synchronize()
    for a, b in ((W1, W2), (M1, M2), (V1, V2)):
        if a is not None:
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_zero_tokens_with_bf16_states():
    """T = 0: the update with a zero gradient, through the element-wise kernel."""
    d_out, d_in = 256, 384
    _, _, w, m, v = _layer(d_out, d_in, 64, "adamw", seed=23)
    hp = default_hparams("adamw", lr=1e-3)
    W, M, V = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step(torch.empty(0, d_out, dtype=torch.bfloat16, device="cuda"),
                     torch.empty(0, d_in, dtype=torch.bfloat16, device="cuda"), W, M, V, None, "adamw", hp, 2, seed=4)
    torch.cuda.synchronize()
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    ref = ostep.apply_update("adamw", np.zeros((d_out, d_in), np.float32), bits(w), bits(m), bits(v), hp, 2, 4, e,
                             "bf16")
    np.testing.assert_array_equal(bits(W.cpu()), ref["W"])
    np.testing.assert_array_equal(bits(M.cpu()), ref["m"])
    np.testing.assert_array_equal(bits(V.cpu()), ref["v"])


@pytest.mark.parametrize("opt", ["adamw", "rmsprop"])
def test_bf16_states_long_token_runs_on_pairs(opt):
    """T = 8192 on CTA pairs (40 pair tiles of 256 x 256)."""
    T, d_out, d_in = 8192, 2048, 1280
    assert fg.launch_shape(d_out, d_in, T)["cluster"] == 2
    dy, x, w, m, v = _layer(d_out, d_in, T, opt, seed=24)
    hp = default_hparams(opt, lr=1e-3)
    W, M, V = w.cuda(), None if m is None else m.cuda(), None if v is None else v.cuda()
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, opt, hp, 4, seed=8)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    _check(opt, dy, x, w, m, v, W.cpu(), None if M is None else M.cpu(), None if V is None else V.cpu(), hp, 4, 8)


def test_llama8b_gate_bf16_states_sampled():
    """Llama-3.1-8B MLP gate (14336 x 4096), T = 4096, AdamW with BF16 states at step 10."""
    wl = WORKLOADS["llama8b-mlp"]
    hp = default_hparams("adamw")
    dy, x = activations(wl, 0, 1)
    w, m, v = layer_state(wl, 0, "adamw")
    m, v = _bf16(m), _bf16(v)
    W, M, V = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, None, "adamw", hp, 10, seed=12)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    d_out, d_in = w.shape
    rows, cols = (np.asarray(a) for a in sample_positions(d_out, d_in, 4096, 9))
    pick = lambda t: bits(t)[rows, cols]
    ref = ostep.fused_step_at("adamw", bits(dy), bits(x), bits(w), bits(m), bits(v), hp, 10, 12, rows, cols,
                              state="bf16")
    e = (rows * d_in + cols).astype(np.uint64)
    rt = moment_rtol(wl.T)
    args = ("adamw", ref["g"], pick(w), pick(m), pick(v), hp, 10, 12, e, rt, "bf16")
    assert_weights(pick(W.cpu()), ref["W"], "W", w_old_bits=pick(w), extra_tol=gradient_sensitivity(*args))
    assert_weights(pick(M.cpu()), ref["m"], "m", w_old_bits=pick(m),
                   extra_tol=gradient_sensitivity(*args, what="m_f32"))
    assert_weights(pick(V.cpu()), ref["v"], "v", w_old_bits=pick(v),
                   extra_tol=gradient_sensitivity(*args, what="v_f32"))
