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


def _run_bench(*args):
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    return subprocess.run([sys.executable, os.path.join(root, "bench.py"), *args], capture_output=True, text=True,
                          cwd=root, timeout=600)


def test_reference_arm_prints_the_contract_line():
    """`--impl reference` times the oracle on a bounded sample and prints one JSON line with the
    contract's keys; the host-buffer e2e of a CPU program moves no bytes over the host link."""
    import json
    r = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--oracle-rows", "8")
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["config"]["workload"].startswith(WORKLOADS["llama8b-mlp"].name)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert cb["blas_threads"]["threads"] >= 1  # the float64 BLAS the oracle's products run on
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_blas_thread_count_without_threadpoolctl(monkeypatch):
    """The GPU machine has no threadpoolctl: the count then comes from numpy's OpenBLAS itself."""
    import sys
    monkeypatch.setitem(sys.modules, "threadpoolctl", None)
    got = bench.blas_threads()
    assert got["threads"] is not None and got["threads"] >= 1 and got["library"] != "unknown"


def test_fewer_than_three_warmup_steps_are_refused():
    r = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0 and "--warmup must be >= 3" in r.stderr


def test_traffic_is_reported_only_for_the_sources_it_was_taken_from(monkeypatch):
    """The committed DRAM traffic per launch stands for the kernel sources whose hash it records;
    once they change, the bench reports no traffic rather than a stale figure."""
    import json
    import os
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")) as f:
        entry = json.load(f)["llama8b-mlp/adamw/fp32"]
    monkeypatch.setattr(bench, "_kernel_source_hash", lambda: entry["source_hash"])
    got = bench._ncu_traffic("llama8b-mlp", "adamw", "fp32")
    assert got == entry["dram_bytes_per_launch"]
    assert got > bench.algorithmic_bytes(WORKLOADS["llama8b-mlp"], "adamw", "fp32", "bf16") / 3
    monkeypatch.setattr(bench, "_kernel_source_hash", lambda: "0" * 16)
    assert bench._ncu_traffic("llama8b-mlp", "adamw", "fp32") is None
    assert bench._ncu_traffic("no-such-workload", "adamw", "fp32") is None


def test_roofline_bound_is_the_slower_unit():
    """The Llama MLP with bf16 operands and FP32 states needs more time at the tensor peak
    (481 GFLOP / 1938 TFLOP/s = 248 us) than at the copy peak (1.325 GB / 6789 GB/s = 195 us):
    tensor-bound.  With E4M3 operands the FP8 peak halves the flop time (124 us) and the same
    W/m/v bytes make it HBM-bound."""
    wl = WORKLOADS["llama8b-mlp"]
    flops = wl.flops_per_step() / 3
    b16 = bench.algorithmic_bytes(wl, "adamw", "fp32", "bf16") / 3
    r = bench.roofline_entry(flops, b16, 0.35, 1938.1, 6789.0, None, {}, "t", "h")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(flops / 0.35e-3 / 1e12 / 1938.1)
    assert r["other"]["bound"] == "hbm" and r["other"]["unit"] == "GB/s"
    b8 = bench.algorithmic_bytes(wl, "adamw", "fp32", "e4m3") / 3
    r8 = bench.roofline_entry(flops, b8, 0.28, 2 * 1938.1, 6789.0, None, {}, "t", "h")
    assert r8["bound"] == "hbm" and r8["unit"] == "GB/s"
    assert r8["achieved"] == pytest.approx(b8 / 0.28e-3 / 1e9) and r8["other"]["bound"] == "tensor"


def test_tensor_peak_follows_the_power_cap():
    """A timed region whose clock samples saw the power cap is held to the sustained GEMM figure;
    any other to the burst figure (and to the fallback when no peaks file gives one)."""
    peaks = {"bf16_tflops": 1938.1, "bf16_tflops_sustained": 1717.2}
    assert bench.tensor_peak_for(peaks, {"reasons": ["sw_power_cap"]}) == (1717.2, "bf16_tflops_sustained")
    assert bench.tensor_peak_for(peaks, {"reasons": []}) == (1938.1, "bf16_tflops")
    assert bench.tensor_peak_for(peaks, None) == (1938.1, "bf16_tflops")
    assert bench.tensor_peak_for({"bf16_tflops": 1900.0}, {"reasons": ["sw_power_cap"]}) == (1900.0, "bf16_tflops")
    assert bench.tensor_peak_for({}, {"reasons": []})[0] == bench.FALLBACK_PEAKS["bf16_tflops"]


def test_oracle_sample_says_what_it_covers():
    """The reference arm's sample names the rows it timed: the whole step for a layer smaller than
    the sample (nothing extrapolated), else each sampled layer's first rows."""
    import json
    r = _run_bench("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["cpu_baseline"]["sample"].startswith("the whole step of tiny")
    assert line["config"]["ms_per_step"] == "measured on the whole step"
