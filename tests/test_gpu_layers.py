"""forge_fused_dw_step_layers: several independent layers per launch (needs a GB300).

The grouped call must give exactly what per-layer forge_fused_dw_step calls give: every element's
update, moment write-back and Philox counter depend only on its own layer, and the tensor core
sums each element's tokens in the same order whatever the tile shape.  Layers run on CTA pairs up
to 16 per launch; small layers, layers without tokens and layers whose tiles are not pairs are
launched one by one inside the same call.
"""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import step as ostep
from tests.compare import assert_moments, assert_weights, gradient_sensitivity, moment_rtol
from tests.helpers import bits, f32
from workloads import Layer, Workload, activations, default_hparams, layer_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


# (d_out, d_in, T): three pair-shaped layers that together fill the GPU, one of them alone too
# small for pairs (512 x 768); a layer whose tiles are not pairs (384 x 512); a layer without tokens
LAYERS = [(2048, 1280, 192), (512, 768, 128), (1024, 1536, 256), (384, 512, 64), (512, 512, 0)]


def _states(opt, shapes, state, seed):
    out = []
    for i, (d_out, d_in, T) in enumerate(shapes):
        wl = Workload("t", (Layer("w", d_out, d_in),), T, 1.0, 1e-3, m_init="absnormal:1e-4", v_init="uniform:1e-6")
        dy, x = activations(wl, 0, 1, seed + i, device="cuda")
        w, m, v = layer_state(wl, 0, opt, seed + i, device="cuda")
        q = None
        if state == "bf16":
            m = None if m is None else m.to(torch.bfloat16)
            v = None if v is None else v.to(torch.bfloat16)
        elif state == "int8":
            g = torch.Generator(device="cuda").manual_seed(seed + i)
            m = None if m is None else torch.randint(-127, 128, (d_out, d_in), generator=g, dtype=torch.int8, device="cuda")
            v = None if v is None else torch.randint(0, 128, (d_out, d_in), generator=g, dtype=torch.int8, device="cuda")
            q = torch.rand(2 * d_out * d_in // 64, generator=g, device="cuda") * 1e-5
        out.append(dict(dy=dy, x=x, w=w, m=m, v=v, q=q, seed=0xC0DE + 17 * i))
    return out


def _clone(layers):
    c = lambda t: None if t is None else t.clone()
    return [dict(L, w=c(L["w"]), m=c(L["m"]), v=c(L["v"]), q=c(L["q"])) for L in layers]


def _same(a, b):
    if a is None:
        return b is None
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("opt, state", [("adamw", "fp32"), ("lion", "fp32"), ("rmsprop", "fp32"), ("sgd", "fp32"),
                                        ("adamw", "bf16"), ("nadam", "bf16"), ("adamw", "int8"), ("adagrad", "int8")])
def test_layers_equal_per_layer_calls_bitwise(opt, state):
    hp = default_hparams(opt, lr=1e-3)
    shapes = [s for s in LAYERS if not (state == "int8" and s[1] % 64)]
    layers = _states(opt, shapes, state, seed=40)
    ref = _clone(layers)
    before = fg.launch_count()
    fg.fused_dw_step_layers([(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], L["seed"]) for L in layers], opt, hp, 3)
    grouped_launches = fg.launch_count() - before
    for L in ref:
        fg.fused_dw_step(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], opt, hp, 3, seed=L["seed"])
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    # the three pair-shaped layers in one launch; the others one launch each
    assert grouped_launches == 1 + (len(shapes) - 3)
    for i, (L, R) in enumerate(zip(layers, ref)):
        for k in ("w", "m", "v", "q"):
            assert _same(L[k], R[k]), f"layer {i} {shapes[i]}: {k} differs"


def test_more_layers_than_one_launch_holds():
    """18 pair-shaped layers: launches of 16 and 2, each layer equal to its own call."""
    hp = default_hparams("adamw", lr=1e-3)
    shapes = [(512, 512, 64)] * 18
    layers = _states("adamw", shapes, "fp32", seed=90)
    ref = _clone(layers)
    before = fg.launch_count()
    fg.fused_dw_step_layers([(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], L["seed"]) for L in layers], "adamw",
                            hp, 2)
    assert fg.launch_count() - before == 2
    for L in ref:
        fg.fused_dw_step(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], "adamw", hp, 2, seed=L["seed"])
    torch.cuda.synchronize()
    for L, R in zip(layers, ref):
        assert _same(L["w"], R["w"]) and _same(L["m"], R["m"]) and _same(L["v"], R["v"])


def test_layers_match_the_oracle():
    """The grouped launch against the oracle directly, every element of two pair-shaped layers."""
    hp = default_hparams("adamw", lr=1e-3)
    shapes = [(2048, 1280, 256), (1024, 1536, 128)]
    layers = _states("adamw", shapes, "fp32", seed=7)
    old = [(bits(L["w"]), f32(L["m"]), f32(L["v"]), bits(L["dy"]), bits(L["x"])) for L in layers]
    fg.fused_dw_step_layers([(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], L["seed"]) for L in layers], "adamw",
                            hp, 5)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    for (d_out, d_in, T), L, (w0, m0, v0, dyb, xb) in zip(shapes, layers, old):
        ref = ostep.fused_step("adamw", dyb, xb, w0, m0, v0, hp, 5, L["seed"])
        e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
        extra = gradient_sensitivity("adamw", ref["g"], w0, m0, v0, hp, 5, L["seed"], e, moment_rtol(T))
        assert_weights(bits(L["w"]), ref["W"], w_old_bits=w0, extra_tol=extra)
        assert_moments(f32(L["m"]), ref["m"], "m", rtol=moment_rtol(T))
        assert_moments(f32(L["v"]), ref["v"], "v", rtol=moment_rtol(T, squared=True))


def test_withheld_stage_in_a_grouped_launch():
    """The failure path of the grouped kernel: a wait runs out, the status reports it, and the
    next grouped call is correct."""
    hp = default_hparams("adamw", lr=1e-3)
    shapes = [(2048, 1280, 256), (1024, 1536, 128)]
    layers = _states("adamw", shapes, "fp32", seed=11)
    ref = _clone(layers)
    fg.set_wait_limit_ns(50_000_000)
    try:
        fg.debug_withhold_next_stage()
        fg.fused_dw_step_layers([(L["dy"], L["x"], L["w"].clone(), L["m"].clone(), L["v"].clone(), None, L["seed"])
                                 for L in layers], "adamw", hp, 2)
        assert fg.sync_status() == 6
    finally:
        fg.set_wait_limit_ns(2_000_000_000)
    fg.fused_dw_step_layers([(L["dy"], L["x"], L["w"], L["m"], L["v"], None, L["seed"]) for L in layers], "adamw", hp, 2)
    for L in ref:
        fg.fused_dw_step(L["dy"], L["x"], L["w"], L["m"], L["v"], None, "adamw", hp, 2, seed=L["seed"])
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    for L, R in zip(layers, ref):
        assert _same(L["w"], R["w"]) and _same(L["m"], R["m"])


@pytest.mark.parametrize("Ts", [(8192, 6144), (8192, 4096)])
def test_int8_layers_with_long_token_runs_equal_per_layer_calls(Ts):
    """INT8 states over long token runs, grouped and per layer: the epilogue stages each block's
    rows in two halves between the operand stages; the grouped call still equals the per-layer
    calls bit for bit."""
    hp = default_hparams("adamw", lr=1e-3)
    shapes = [(2048, 1280, Ts[0]), (1024, 1536, Ts[1])]
    layers = _states("adamw", shapes, "int8", seed=61)
    ref = _clone(layers)
    before = fg.launch_count()
    fg.fused_dw_step_layers([(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], L["seed"]) for L in layers], "adamw",
                            hp, 4)
    assert fg.launch_count() - before == 1
    for L in ref:
        fg.fused_dw_step(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], "adamw", hp, 4, seed=L["seed"])
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    for i, (L, R) in enumerate(zip(layers, ref)):
        for k in ("w", "m", "v", "q"):
            assert _same(L[k], R[k]), f"layer {i} {shapes[i]}: {k} differs"


@pytest.mark.parametrize("state", ["fp32", "int8"])
def test_grouped_launch_with_a_split_tail_equals_per_layer_calls(state):
    """Two 2048 x 1280 layers: 40 pair tiles each, one wave on its own; together 80 tiles, so the
    grouped launch runs its last 4 as half tiles.  The sums do not depend on the tile shape, so
    every byte still equals the per-layer calls'."""
    hp = default_hparams("adamw", lr=1e-3)
    shapes = [(2048, 1280, 320), (2048, 1280, 192)]
    layers = _states("adamw", shapes, state, seed=77)
    ref = _clone(layers)
    before = fg.launch_count()
    fg.fused_dw_step_layers([(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], L["seed"]) for L in layers], "adamw",
                            hp, 2)
    assert fg.launch_count() - before == 1
    for L in ref:
        fg.fused_dw_step(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], "adamw", hp, 2, seed=L["seed"])
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    for i, (L, R) in enumerate(zip(layers, ref)):
        for k in ("w", "m", "v", "q"):
            assert _same(L[k], R[k]), f"layer {i}: {k} differs"


def test_split_tail_across_a_layer_boundary():
    """1536 x 3328 (78 pair tiles) and 256 x 512 (2): the grouped launch's 80 tiles end on a split
    tail of 4 tiles, two from each layer, so half tiles of both layers run in the last wave."""
    hp = default_hparams("adamw", lr=1e-3)
    shapes = [(1536, 3328, 128), (256, 512, 192)]
    layers = _states("adamw", shapes, "fp32", seed=83)
    ref = _clone(layers)
    before = fg.launch_count()
    fg.fused_dw_step_layers([(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], L["seed"]) for L in layers], "adamw",
                            hp, 3)
    assert fg.launch_count() - before == 1
    for L in ref:
        fg.fused_dw_step(L["dy"], L["x"], L["w"], L["m"], L["v"], L["q"], "adamw", hp, 3, seed=L["seed"])
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    for i, (L, R) in enumerate(zip(layers, ref)):
        for k in ("w", "m", "v"):
            assert _same(L[k], R[k]), f"layer {i}: {k} differs"
