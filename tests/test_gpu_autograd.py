"""`ForgeLinear` (PyTorch autograd integration) on the GPU: its backward equals the library's calls.

The fused step itself is checked against the oracle elsewhere; here the layer's backward must make
exactly the calls a user would make by hand (same step count, seed and state), so W, the moments
and the input gradient are compared bit for bit with those calls, and dX once more with the oracle.
"""
import pytest
import torch

import backward_optimizer_gb300 as fg
from backward_optimizer_gb300.autograd import ForgeLinear
from oracle import backward as obw
from tests.compare import assert_bf16_sum
from tests.helpers import bits
from workloads import default_hparams, normal_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def _same(a, b):
    if a is None or b is None:
        return a is None and b is None
    return torch.equal(a.view(torch.int8) if a.dtype == torch.int8 else a.contiguous().view(torch.uint8),
                       b.view(torch.int8) if b.dtype == torch.int8 else b.contiguous().view(torch.uint8))


def _snapshot(layer):
    return [None if t is None else t.detach().clone() for t in (layer.weight, layer.m, layer.v, layer.qscales)]


@pytest.mark.parametrize("opt, state", [("adamw", "fp32"), ("lion", "bf16"), ("adamw", "int8"), ("sgd", "fp32")])
def test_backward_is_the_fused_layer_backward(opt, state):
    """Two training steps through autograd, x [2, 160, d_in] (T = 320, a ragged token tail)."""
    d_in, d_out, seed = 512, 384, 7
    hp = default_hparams(opt, lr=1e-2)
    layer = ForgeLinear(d_in, d_out, opt, hp, state=state, seed=seed)
    layer.weight.data.copy_(normal_bf16((d_out, d_in), 2e-2, seed=1).cuda())
    for step in (1, 2):
        x = normal_bf16((2, 160, d_in), 1.0, seed=10 + step).cuda().requires_grad_(True)
        dy = normal_bf16((2, 160, d_out), 1e-3, seed=20 + step).cuda()
        W, m, v, q = _snapshot(layer)
        w_before = W.clone()
        layer(x).backward(dy)
        dX = torch.empty(320, d_in, dtype=torch.bfloat16, device="cuda")
        fg.linear_backward(dy.reshape(320, d_out), x.detach().reshape(320, d_in), W, m, v, q, dX, opt, hp, step, seed)
        torch.cuda.synchronize()
        assert fg.sync_status() == 0
        assert layer.weight.grad is None and layer.step == step + 1
        for got, want in zip((layer.weight, layer.m, layer.v, layer.qscales), (W, m, v, q)):
            assert _same(got, want)
        assert x.grad.shape == x.shape and _same(x.grad.reshape(320, d_in), dX)
        assert_bf16_sum(bits(x.grad.reshape(320, d_in)), obw.dx_f32(bits(dy.reshape(320, d_out)), bits(w_before)),
                        d_out)


def test_input_without_grad_takes_the_weight_step_only():
    """x that does not require grad: the fused step alone (no dX), same result as fused_dw_step."""
    layer = ForgeLinear(256, 256, "adamw", default_hparams("adamw", lr=1e-2), seed=3)
    x = normal_bf16((192, 256), 1.0, seed=30).cuda()
    dy = normal_bf16((192, 256), 1e-3, seed=31).cuda()
    W, m, v, _ = _snapshot(layer)
    before = fg.launch_count()
    layer(x).backward(dy)
    torch.cuda.synchronize()
    assert fg.launch_count() - before == 1
    fg.fused_dw_step(dy, x, W, m, v, None, "adamw", layer.hp, 1, 3)
    torch.cuda.synchronize()
    assert x.grad is None
    assert _same(layer.weight, W) and _same(layer.m, m) and _same(layer.v, v)


def test_one_backward_per_forward():
    layer = ForgeLinear(256, 128, "sgd_momentum", default_hparams("sgd_momentum"), seed=4)
    x = normal_bf16((64, 256), 1.0, seed=40).cuda().requires_grad_(True)
    y = layer(x).float().sum()
    y.backward(retain_graph=True)
    with pytest.raises(RuntimeError, match="one backward per forward"):
        y.backward()
    torch.cuda.synchronize()
    assert layer.step == 2


def test_no_grad_forward_leaves_the_layer_alone():
    layer = ForgeLinear(128, 128, "adamw", seed=5)
    x = normal_bf16((64, 128), 1.0, seed=50).cuda()
    with torch.no_grad():
        y = layer(x)
    ref = torch.nn.functional.linear(x, layer.weight)
    assert torch.equal(y, ref) and layer.step == 1
