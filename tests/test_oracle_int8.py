"""Pins for the oracle's INT8 block-64 codec (CPU only)."""
import numpy as np

from oracle import int8_block


def _blocks(seed, n=512):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, 64)).astype(np.float32) * np.float32(10.0) ** rng.integers(-8, 3, (n, 1))
    return x.astype(np.float32)


def test_roundtrip_error_at_most_half_a_step():
    x = _blocks(0)
    q, s = int8_block.quantize(x)
    xr = int8_block.dequantize(q, s)
    err = np.abs(xr.astype(np.float64) - x.astype(np.float64))
    # half a quantisation step, plus the binary32 roundings of x/s and q*s
    bound = s.astype(np.float64) * (0.5 + 1e-5)  # s: (n, 1), one scale per block
    assert np.all(err <= bound)


def test_absmax_element_maps_to_full_code():
    x = _blocks(1)
    q, s = int8_block.quantize(x)
    k = np.argmax(np.abs(x), axis=1)
    top = q[np.arange(x.shape[0]), k].astype(np.int64)
    assert np.all(np.abs(top) == 127)
    assert np.all(np.sign(top) == np.sign(x[np.arange(x.shape[0]), k]))
    assert np.all(np.abs(q.astype(np.int64)) <= 127)


def test_zero_block_and_single_value():
    x = np.zeros((2, 64), np.float32)
    x[1, 5] = -3.0
    q, s = int8_block.quantize(x)
    assert s[0] == 0 and np.all(q[0] == 0)
    assert np.all(int8_block.dequantize(q, s)[0] == 0)
    assert q[1, 5] == -127 and np.all(np.delete(q[1], 5) == 0)
    assert int8_block.dequantize(q, s)[1, 5] == np.float32(-3.0) / np.float32(127) * np.float32(127)


def test_codes_are_nearest_by_brute_force():
    """Each code is the integer in [-127, 127] whose binary32 ratio x/s is nearest (ties to even)."""
    x = _blocks(2, n=64)
    q, s = int8_block.quantize(x)
    cand = np.arange(-127, 128, dtype=np.float64)
    for b in range(x.shape[0]):
        ratio = (x[b] / s[b]).astype(np.float32).astype(np.float64)
        d = np.abs(ratio[:, None] - cand[None, :])
        best = cand[np.argmin(d, axis=1)]
        ties = np.isclose(np.sort(d, axis=1)[:, 0], np.sort(d, axis=1)[:, 1], rtol=0, atol=0)
        ok = (q[b].astype(np.float64) == best) | ties
        assert np.all(ok)


def test_blocks_are_64_consecutive_elements_of_a_row():
    x = np.ones((1, 128), np.float32)
    x[0, 64:] *= 1000
    q, s = int8_block.quantize(x)
    assert s.shape == (1, 2)
    assert np.all(q == 127)
    assert s[0, 1] == np.float32(1000) / np.float32(127)
