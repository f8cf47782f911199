"""Failure detection on the GPU without a fault: a bounded wait is made to run out (the producer
withholds one pipeline stage that nothing else will fill), the kernel reports FORGE_ERR_TIMEOUT
through the device status word and returns, and the context stays usable (needs a GB300)."""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import step as ostep
from tests.compare import assert_moments, assert_weights, gradient_sensitivity, moment_rtol
from tests.helpers import bits, f32
from workloads import Layer, Workload, activations, default_hparams, layer_state

pytestmark = pytest.mark.gpu

TIMEOUT = 6  # FORGE_ERR_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()
    assert fg.sync_status() == 0
    fg.set_wait_limit_ns(50_000_000)  # 50 ms
    yield
    fg.set_wait_limit_ns(2_000_000_000)
    fg.sync_status()


def _layer(d_out, d_in, T):
    wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
    dy, x = activations(wl, 0, 1, 3)
    w, m, v = layer_state(wl, 0, "adamw", 3)
    return dy, x, w, m, v


# (2048, 1280): a CTA pair, over a long and a short token run; (1152, 2560): one CTA, 128 x 256;
# (1536, 1536): one CTA, 128 x 128; (384, 384): one CTA, 128 x 64
@pytest.mark.parametrize("d_out, d_in, T", [(2048, 1280, 8192), (2048, 1280, 512), (1152, 2560, 512), (1536, 1536, 512),
                                            (384, 384, 512)])
def test_withheld_stage_times_out_and_context_survives(d_out, d_in, T):
    dy, x, w, m, v = _layer(d_out, d_in, T)
    hp = default_hparams("adamw", lr=1e-3)
    D, X = dy.cuda(), x.cuda()
    fg.debug_withhold_next_stage()
    fg.fused_dw_step(D, X, w.cuda(), m.cuda(), v.cuda(), None, "adamw", hp, 2, seed=1)
    assert fg.sync_status() == TIMEOUT
    assert fg.sync_status() == 0  # the status word was cleared by the read
    # the next call on the same context is complete and correct
    W, M, V = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step(D, X, W, M, V, None, "adamw", hp, 2, seed=1)
    assert fg.sync_status() == 0
    ref = ostep.fused_step("adamw", bits(dy), bits(x), bits(w), f32(m), f32(v), hp, 2, 1)
    rt = moment_rtol(T)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity("adamw", ref["g"], bits(w), f32(m), f32(v), hp, 2, 1, e, rt)
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    assert_moments(f32(M), ref["m"], "m", rtol=rt)
    assert_moments(f32(V), ref["v"], "v", rtol=moment_rtol(T, squared=True))


def test_withheld_stage_in_the_e4m3_step():
    from oracle import fp8
    from workloads import activations_fp8
    T, d_out, d_in = 512, 2048, 1280
    wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
    dyq, s_dy, xq, s_x = activations_fp8(wl, 0, 1, 3)
    w, m, v = layer_state(wl, 0, "adamw", 3)
    hp = default_hparams("adamw", lr=1e-3)
    D, X = dyq.cuda(), xq.cuda()
    fg.debug_withhold_next_stage()
    fg.fused_dw_step_e4m3(D, X, s_dy, s_x, w.cuda(), m.cuda(), v.cuda(), None, "adamw", hp, 2, seed=1)
    assert fg.sync_status() == TIMEOUT
    W, M, V = w.cuda(), m.cuda(), v.cuda()
    fg.fused_dw_step_e4m3(D, X, s_dy, s_x, W, M, V, None, "adamw", hp, 2, seed=1)
    assert fg.sync_status() == 0
    ref = fp8.fused_step_fp8("adamw", dyq.numpy(), xq.numpy(), s_dy, s_x, bits(w), f32(m), f32(v), hp, 2, 1)
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    extra = gradient_sensitivity("adamw", ref["g"], bits(w), f32(m), f32(v), hp, 2, 1, e, moment_rtol(T))
    assert_weights(bits(W), ref["W"], w_old_bits=bits(w), extra_tol=extra)
    assert_moments(f32(M), ref["m"], "m")


@pytest.mark.parametrize("kind", ["dx", "dw"])
def test_withheld_stage_in_the_gemms(kind):
    """The input-gradient and weight-gradient GEMMs run the same pipeline and report the same way
    (both on CTA pairs: dX 2048 x 1280 and dW 2048 x 1280 have 40 pair tiles)."""
    from oracle import backward as obw
    from tests.compare import assert_bf16_sum
    d_out, d_in, T = (512, 1280, 2048) if kind == "dx" else (2048, 1280, 512)
    dy, x, w, _, _ = _layer(d_out, d_in, T)
    D, X, Wd = dy.cuda(), x.cuda(), w.cuda()
    for attempt in range(2):
        if attempt == 0:
            fg.debug_withhold_next_stage()
        if kind == "dx":
            assert fg.dx_launch_shape(T, d_out, d_in)["cluster"] == 2
            out = torch.empty(T, d_in, dtype=torch.bfloat16, device="cuda")
            fg.dx_gemm(D, Wd, out)
        else:
            assert fg.launch_shape(d_out, d_in, T)["cluster"] == 2
            out = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
            fg.dw_gemm(D, X, out)
        assert fg.sync_status() == (TIMEOUT if attempt == 0 else 0)
    if kind == "dx":
        assert_bf16_sum(bits(out), obw.dx_f32(bits(dy), bits(w)), d_out)
    else:
        assert_moments(out.cpu().numpy(), ostep.dw(bits(dy), bits(x)), "dW")
