"""The benchmark's byte accounting for the HBM side of the roofline (CPU only)."""
import pytest

import bench
from workloads import WORKLOADS, Layer, Workload


def _one_layer(T=0):
    return Workload("t", (Layer("w", 128, 64),), T, 1.0, 1e-3)


@pytest.mark.parametrize("opt, state, per_element", [
    ("adamw", "fp32", 20.0),            # W 2+2, m 4+4, v 4+4
    ("adamw", "bf16", 12.0),            # W 2+2, m 2+2, v 2+2
    ("adamw", "int8", 4.0 + 2 * (2 + 8 / 64)),  # W 2+2, codes 1+1 and a 4-byte scale per 64 each way, twice
    ("lion", "fp32", 12.0),             # one moment
    ("rmsprop", "fp32", 12.0),
    ("sgd", "fp32", 4.0),               # no state
])
def test_per_element_bytes(opt, state, per_element):
    assert bench.algorithmic_bytes(_one_layer(), opt, state, "bf16") == pytest.approx(128 * 64 * per_element)


def test_operands_read_once_at_their_width():
    wl = _one_layer(T=256)
    base = bench.algorithmic_bytes(_one_layer(), "sgd", "fp32", "bf16")
    assert bench.algorithmic_bytes(wl, "sgd", "fp32", "bf16") - base == 256 * (128 + 64) * 2
    assert bench.algorithmic_bytes(wl, "sgd", "fp32", "e4m3") - base == 256 * (128 + 64) * 1


def test_llama_mlp_launch_bytes():
    """The figure the profile summary derives: 1.325 GB per Llama-8B MLP launch (AdamW, FP32 states)."""
    wl = WORKLOADS["llama8b-mlp"]
    assert bench.algorithmic_bytes(wl, "adamw", "fp32", "bf16") / 3 == pytest.approx(1.3254e9, rel=1e-4)
