"""`ForgeLinear` host logic on the CPU: buffers per optimizer and state format, argument checks and
the one-backward-per-forward guard (no kernel runs here)."""
import pytest
import torch

from backward_optimizer_gb300.autograd import ForgeLinear


@pytest.mark.parametrize("opt, m, v", [("adamw", True, True), ("lion", True, False), ("adagrad", False, True),
                                       ("sgd", False, False)])
@pytest.mark.parametrize("state, dtype", [("fp32", torch.float32), ("bf16", torch.bfloat16), ("int8", torch.int8)])
def test_buffers(opt, m, v, state, dtype):
    layer = ForgeLinear(128, 64, opt, state=state, device="cpu")
    assert layer.weight.dtype == torch.bfloat16 and tuple(layer.weight.shape) == (64, 128)
    assert not layer.weight.requires_grad
    for buf, used in ((layer.m, m), (layer.v, v)):
        assert (buf is not None) == used
        if used:
            assert buf.dtype == dtype and tuple(buf.shape) == (64, 128) and not buf.any()
    if state == "int8" and (m or v):
        assert layer.qscales.shape == (2 * 64 * 128 // 64,)
    else:
        assert layer.qscales is None
    assert dict(layer.named_buffers()).keys() == {k for k, u in (("m", m), ("v", v)) if u} | (
        {"qscales"} if state == "int8" and (m or v) else set())


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        ForgeLinear(64, 64, "adam", device="cpu")
    with pytest.raises(ValueError):
        ForgeLinear(64, 64, "adamw", state="fp16", device="cpu")
    layer = ForgeLinear(64, 64, device="cpu")
    with pytest.raises(TypeError):
        layer(torch.zeros(4, 64))


def test_no_grad_forward_is_linear():
    layer = ForgeLinear(64, 32, device="cpu")
    x = torch.randn(5, 64).to(torch.bfloat16)
    with torch.no_grad():
        assert torch.equal(layer(x), torch.nn.functional.linear(x, layer.weight))
    assert layer.step == 1


def test_second_backward_is_refused_before_any_call():
    layer = ForgeLinear(64, 32, device="cpu")
    with pytest.raises(RuntimeError, match="one backward per forward"):
        layer._step_once(None, None, None)
