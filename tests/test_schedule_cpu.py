"""The persistent tile order of the tile kernel (csrc/schedule.h), compiled for the host with g++."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def report(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    exe = str(tmp_path_factory.mktemp("sched") / "schedule_check")
    subprocess.run([gxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I",
                    os.path.join(ROOT, "backward_optimizer_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "c", "schedule_check.cpp"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout
    return dict((l.split()[0], l.split()[1:]) for l in out.stdout.splitlines())


def test_every_tile_order_is_a_bijection(report):
    assert report["bijection_failures"] == ["0"]


@pytest.mark.parametrize("case, raster_cols, group", [
    # X (the smaller operand) resident: all 16 tile columns per group, tile rows stream past
    ("llama_gate", 1, 16),
    # dY resident: all 16 tile rows per group
    ("llama_down", 0, 16),
    # equal operands: rows grouped, as many 4 MiB dY blocks as fit in 48 MiB
    ("qwen_q", 0, 12), ("qwen_k", 0, 4), ("qwen_gate", 1, 12), ("qwen_down", 0, 12)])
def test_the_smaller_operand_is_kept_resident(report, case, raster_cols, group):
    assert report[case] == ["raster_cols", str(raster_cols), "group", str(group)]
