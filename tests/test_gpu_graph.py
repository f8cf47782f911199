"""The library's calls inside a captured CUDA graph (needs a GB300).

Small layers are bound by the host's launch path; capturing a step's calls once and replaying the
graph removes it.  A replay must give exactly what the same calls give when issued one by one: the
calls encode their tensor maps on the host and pass them by value, and nothing in them synchronises,
so capture records the same launches.  The first call on a device sets the device up (symbol
address, kernel attributes), so each test makes one call before capturing.
"""
import pytest
import torch

import backward_optimizer_gb300 as fg
from workloads import Layer, Workload, activations, activations_fp8, default_hparams, layer_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def _state(d_out, d_in, T, seed):
    wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
    dy, x = activations(wl, 0, 1, seed, device="cuda")
    w, m, v = layer_state(wl, 0, "adamw", seed, device="cuda")
    return wl, dy, x, w, m, v


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16)) if a.dtype == torch.bfloat16 else torch.equal(a, b)


@pytest.mark.parametrize("d_out, d_in, T", [(512, 256, 256), (1024, 1024, 512)])
def test_replayed_layer_backward_equals_eager(d_out, d_in, T):
    """dX then the fused step, three times: graph replays against eager calls, bit for bit."""
    wl, dy, x, w, m, v = _state(d_out, d_in, T, seed=1)
    hp = default_hparams("adamw", lr=1e-3)
    W1, M1, V1, dX1 = w.clone(), m.clone(), v.clone(), torch.empty(T, d_in, dtype=torch.bfloat16, device="cuda")
    W2, M2, V2, dX2 = w.clone(), m.clone(), v.clone(), torch.empty_like(dX1)
    # set up the device (and load the kernels) before capture, on throwaway copies
    fg.linear_backward(dy, x, w.clone(), m.clone(), v.clone(), None, torch.empty_like(dX1), "adamw", hp, 2, seed=3)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side), torch.cuda.graph(graph):
        fg.linear_backward(dy, x, W1, M1, V1, None, dX1, "adamw", hp, 2, seed=3)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        graph.replay()
        fg.linear_backward(dy, x, W2, M2, V2, None, dX2, "adamw", hp, 2, seed=3)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    for a, b in ((W1, W2), (M1, M2), (V1, V2), (dX1, dX2)):
        assert _same(a, b)
    assert not torch.equal(W1, w)  # the replays did update the weights


def test_replayed_e4m3_step_equals_eager():
    wl = Workload("t", (Layer("w", 512, 768),), 320, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
    dyq, s_dy, xq, s_x = activations_fp8(wl, 0, 1, 2, device="cuda")
    w, m, v = layer_state(wl, 0, "adamw", 2, device="cuda")
    hp = default_hparams("adamw", lr=1e-3)
    W1, M1, V1 = w.clone(), m.clone(), v.clone()
    W2, M2, V2 = w.clone(), m.clone(), v.clone()
    fg.fused_dw_step_e4m3(dyq, xq, s_dy, s_x, w.clone(), m.clone(), v.clone(), None, "adamw", hp, 5, seed=4)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side), torch.cuda.graph(graph):
        fg.fused_dw_step_e4m3(dyq, xq, s_dy, s_x, W1, M1, V1, None, "adamw", hp, 5, seed=4)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        graph.replay()
        fg.fused_dw_step_e4m3(dyq, xq, s_dy, s_x, W2, M2, V2, None, "adamw", hp, 5, seed=4)
    torch.cuda.synchronize()
    for a, b in ((W1, W2), (M1, M2), (V1, V2)):
        assert _same(a, b)
