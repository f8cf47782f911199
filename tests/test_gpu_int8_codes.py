"""INT8 requantisation pinned bit for bit through the kernels (needs a GB300).

The other INT8 parity tests allow codes to differ by one, because the oracle computes the update in
float64 and the kernels in binary32, so a moment that lands next to a rounding boundary can fall on
either side.  Here every new moment is exact on both sides: the states start at zero, the decays
are 1/2, weight decay is 0, and dY and X hold small integers, so dW = dY^T X is an exact integer
whatever the summation order.  The new moments are then g/2, g or RN(g^2)/2 on both sides, and the
block scale RN(absmax / 127) and every code rne(RN(x / s)) must agree exactly: this pins the
kernels' division, rounding and clamping of the codes against the oracle's definition.
"""
import numpy as np
import pytest
import torch

import backward_optimizer_gb300 as fg
from oracle import fp8, step as ostep
from tests.helpers import bits
from workloads import Hparams, OPTIMIZERS, random_codes

pytestmark = pytest.mark.gpu

HALF = Hparams(lr=1e-3, beta1=0.5, beta2=0.5, eps=1e-8, weight_decay=0.0, momentum=0.9, alpha=0.5)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fg.build()
    fg.lib()


def _integer_bf16(shape, seed):
    """Integers in [-15, 15] as bfloat16 (exact)."""
    return (random_codes(shape, seed, -15, 15).to(torch.float32)).to(torch.bfloat16)


def _case(opt, d_out, d_in, T, seed):
    dy = _integer_bf16((T, d_out), seed)
    x = _integer_bf16((T, d_in), seed + 1)
    w = (torch.randn(d_out, d_in, generator=torch.Generator().manual_seed(seed + 2)) * 0.02).to(torch.bfloat16)
    zeros = np.zeros((d_out, d_in), np.int8)
    nblk = d_out * d_in // 64
    return dy, x, w, zeros, np.zeros((d_out, d_in // 64), np.float32), nblk


def _check(opt, M, V, Q, ref, nblk, g):
    # the construction's premise, on the oracle's side: new moments g/2, g, RN(g^2)/2 or RN(g^2)
    exact_m = {"sgd_momentum": g}.get(opt, g / 2)
    g2 = (g.astype(np.float64) ** 2).astype(np.float32)
    exact_v = g2 if opt == "adagrad" else g2 / 2
    if ref["m_f32"] is not None:
        assert np.array_equal(ref["m_f32"], exact_m.astype(np.float32))
    if ref["v_f32"] is not None:
        assert np.array_equal(ref["v_f32"], exact_v)
    q = Q.cpu().numpy()
    for got, codes, scales, sl in ((M, ref["m"], ref["m_scales"], slice(0, nblk)),
                                   (V, ref["v"], ref["v_scales"], slice(nblk, 2 * nblk))):
        if codes is None:
            continue
        assert np.array_equal(got.cpu().numpy(), codes), f"{opt}: {np.sum(got.cpu().numpy() != codes)} codes differ"
        assert np.array_equal(q[sl].view(np.uint32), scales.ravel().astype(np.float32).view(np.uint32)), \
            f"{opt}: scales differ"


def _exact_gradient(dy, x):
    g = ostep.dw(bits(dy), bits(x))
    assert np.array_equal(g, np.rint(g)) and np.abs(g).max() < 2 ** 24
    return g


# (d_out, d_in, T): a CTA pair on 256 x 256 tiles (40 pair tiles); one CTA on 128 x 256 tiles (90);
# a CTA pair over a long token run (T = 8192)
# the last: 80 pair tiles, whose last 4 run as 8 half tiles (two warps per 64-column block)
SHAPES = [(2048, 1280, 256, (256, 256)), (1152, 2560, 192, (128, 256)), (2048, 1280, 8192, (256, 256)),
          (4096, 1280, 128, (256, 256))]


@pytest.mark.parametrize("opt", [o for o in OPTIMIZERS if o != "sgd"])
@pytest.mark.parametrize("d_out, d_in, T, tile", SHAPES)
def test_fused_int8_codes_are_exact(opt, d_out, d_in, T, tile):
    got = fg.launch_shape(d_out, d_in, T)
    assert (got["tile_rows"], got["tile_cols"]) == tile
    dy, x, w, zeros, zscales, nblk = _case(opt, d_out, d_in, T, seed=10 * OPTIMIZERS.index(opt))
    g = _exact_gradient(dy, x)
    W, M, V = w.cuda(), torch.from_numpy(zeros).cuda(), torch.from_numpy(zeros).cuda()
    Q = torch.zeros(2 * nblk, dtype=torch.float32, device="cuda")
    fg.fused_dw_step(dy.cuda(), x.cuda(), W, M, V, Q, opt, HALF, 1, seed=1)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    ref = ostep.apply_update(opt, g, bits(w), zeros, zeros, HALF, 1, 1, e, "int8", zscales, zscales)
    _check(opt, M, V, Q, ref, nblk, g)


@pytest.mark.parametrize("opt", ["adamw", "adagrad", "sgd_momentum"])
def test_two_phase_int8_codes_are_exact(opt):
    d_out, d_in, T = 256, 512, 128
    dy, x, w, zeros, zscales, nblk = _case(opt, d_out, d_in, T, seed=77)
    g = _exact_gradient(dy, x)
    W, M, V = w.cuda(), torch.from_numpy(zeros).cuda(), torch.from_numpy(zeros).cuda()
    Q = torch.zeros(2 * nblk, dtype=torch.float32, device="cuda")
    fg.opt_step(torch.from_numpy(g).cuda(), W, M, V, Q, opt, HALF, 1, seed=1)
    torch.cuda.synchronize()
    e = np.arange(d_out * d_in, dtype=np.uint64).reshape(d_out, d_in)
    ref = ostep.apply_update(opt, g, bits(w), zeros, zeros, HALF, 1, 1, e, "int8", zscales, zscales)
    _check(opt, M, V, Q, ref, nblk, g)


def _e4m3_codes(t):
    """Small integers (|v| <= 15, exact in E4M3) as E4M3 codes."""
    return t.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


@pytest.mark.parametrize("opt", ["adamw", "lion", "adagrad"])
@pytest.mark.parametrize("d_out, d_in, T, tile", [SHAPES[0], SHAPES[2]])
def test_fused_int8_codes_are_exact_with_e4m3_operands(opt, d_out, d_in, T, tile):
    """The same construction through the E4M3 mainloop: integer codes with scales 1 keep g exact."""
    got = fg.launch_shape(d_out, d_in, T)
    assert (got["tile_rows"], got["tile_cols"]) == tile
    dy, x, w, zeros, zscales, nblk = _case(opt, d_out, d_in, T, seed=200 + OPTIMIZERS.index(opt))
    dyq, xq = _e4m3_codes(dy), _e4m3_codes(x)
    g = fp8.dw_fp8(dyq.numpy(), xq.numpy(), 1.0, 1.0)
    assert np.array_equal(g, _exact_gradient(dy, x))
    W, M, V = w.cuda(), torch.from_numpy(zeros).cuda(), torch.from_numpy(zeros).cuda()
    Q = torch.zeros(2 * nblk, dtype=torch.float32, device="cuda")
    fg.fused_dw_step_e4m3(dyq.cuda(), xq.cuda(), 1.0, 1.0, W, M, V, Q, opt, HALF, 1, seed=1)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    ref = fp8.fused_step_fp8(opt, dyq.numpy(), xq.numpy(), 1.0, 1.0, bits(w), zeros, zeros, HALF, 1, 1, "int8",
                             zscales, zscales)
    _check(opt, M, V, Q, ref, nblk, g)


def _random_int8_state(shape, seed):
    """Random signed m codes and non-negative v codes with positive block scales."""
    g = torch.Generator().manual_seed(seed)
    m = torch.randint(-127, 128, shape, generator=g, dtype=torch.int8)
    v = torch.randint(0, 128, shape, generator=g, dtype=torch.int8)
    n = shape[0] * shape[1] // 64
    q = torch.cat([torch.rand(n, generator=g) * 1e-5, torch.rand(n, generator=g) * 1e-8])
    return m, v, q


@pytest.mark.parametrize("opt", [o for o in OPTIMIZERS if o != "sgd"])
@pytest.mark.parametrize("d_out, d_in, T, tile", SHAPES)
def test_fused_int8_equals_two_phase_bitwise(opt, d_out, d_in, T, tile):
    """Random states and operands: the fused kernel codes from the block's reciprocal (and the
    IEEE division near rounding boundaries), the two-phase kernel always divides.  Same mainloop,
    same moments, so weights, codes and scales must agree bit for bit."""
    got = fg.launch_shape(d_out, d_in, T)
    assert (got["tile_rows"], got["tile_cols"]) == tile
    from workloads import normal_bf16
    dy = normal_bf16((T, d_out), 1e-3, seed=300 + T).cuda()
    x = normal_bf16((T, d_in), 1.0, seed=301 + T).cuda()
    w = normal_bf16((d_out, d_in), 2e-2, seed=302).cuda()
    m, v, q = (t.cuda() for t in _random_int8_state((d_out, d_in), 303 + OPTIMIZERS.index(opt)))
    hp = Hparams(lr=1e-3)
    W1, M1, V1, Q1 = w.clone(), m.clone(), v.clone(), q.clone()
    W2, M2, V2, Q2 = w.clone(), m.clone(), v.clone(), q.clone()
    fg.fused_dw_step(dy, x, W1, M1, V1, Q1, opt, hp, 3, seed=4)
    dW = torch.empty(d_out, d_in, dtype=torch.float32, device="cuda")
    fg.dw_gemm(dy, x, dW)
    fg.opt_step(dW, W2, M2, V2, Q2, opt, hp, 3, seed=4)
    torch.cuda.synchronize()
    assert fg.sync_status() == 0
    assert torch.equal(W1.view(torch.int16), W2.view(torch.int16))
    assert torch.equal(M1, M2) and torch.equal(V1, V2)
    assert torch.equal(Q1.view(torch.int32), Q2.view(torch.int32))
