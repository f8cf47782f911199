"""Pins for the oracle's Philox4x32-10 and its SR bit stream (CPU only)."""
import os

import numpy as np
import pytest

from oracle import philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(w, 16) for w in line.split()])
    return rows


@pytest.mark.parametrize("row", _kat_rows())
def test_known_answer_vectors(row):
    ctr = [np.array([w], dtype=np.uint32) for w in row[0:4]]
    out = philox.philox4x32(ctr, (row[4], row[5]))
    assert [int(o[0]) for o in out] == row[6:10]


def test_round_count_matters():
    z = [np.zeros(1, np.uint32)] * 4
    assert [int(o[0]) for o in philox.philox4x32(z, (0, 0), rounds=7)] != _kat_rows()[0][6:10]


def test_bijective_on_sampled_counters():
    rng = np.random.default_rng(1)
    ctr = rng.integers(0, 2**32, size=(4, 200_000), dtype=np.uint64).astype(np.uint32)
    ctr[1, :] = 7  # vary only words 0, 2, 3 -> distinct inputs must stay distinct
    ctr = np.unique(ctr, axis=1)
    out = philox.philox4x32(ctr, (123, 456))
    assert np.unique(out, axis=1).shape[1] == ctr.shape[1]


def test_sr_bits_uniform_chi_square():
    e = np.arange(1 << 20, dtype=np.uint64)
    r = philox.sr_bits(seed=0, step=1, e=e)
    assert r.max() < 65536
    hist = np.bincount((r >> 8).astype(np.int64), minlength=256)  # 256 bins of the top byte
    expected = e.size / 256
    chi2 = float(((hist - expected) ** 2 / expected).sum())
    # 255 degrees of freedom: mean 255, sd ~22.6; 400 is beyond 6 sd.
    assert chi2 < 400, chi2
    lo = np.bincount((r & 0xFF).astype(np.int64), minlength=256)
    assert float(((lo - expected) ** 2 / expected).sum()) < 400


def test_sr_bits_layout_eight_elements_per_call():
    """Elements 8j..8j+7 take the halves of the four words of one Philox call."""
    seed, step, j = 0x1234_5678_9ABC, 17, 5
    e = np.arange(8 * j, 8 * j + 8, dtype=np.uint64)
    r = philox.sr_bits(seed, step, e)
    ctr = [np.array([j], np.uint32), np.array([0], np.uint32),
           np.array([step], np.uint32), np.array([0], np.uint32)]
    words = philox.philox4x32(ctr, (seed & 0xFFFFFFFF, seed >> 32))[:, 0]
    expect = []
    for w in words:
        expect += [int(w) & 0xFFFF, int(w) >> 16]
    assert r.tolist() == expect


def test_sr_bits_depend_on_seed_step_and_index():
    e = np.arange(4096, dtype=np.uint64)
    a = philox.sr_bits(1, 1, e)
    assert not np.array_equal(a, philox.sr_bits(2, 1, e))
    assert not np.array_equal(a, philox.sr_bits(1, 2, e))
    assert not np.array_equal(a, philox.sr_bits(1, 1, e + 8))
    assert np.array_equal(a, philox.sr_bits(1, 1, e))
