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


def test_groups_of_rows_sweep_one_column_at_a_time(report):
    # 20 x 4 tiles in groups of 8 rows: tiles 0..7 are rows 0..7 of column 0, tile 8 starts column 1;
    # the first group ends at tile 31 (row 7, column 3); the last group has the 4 rows 16..19
    assert report["rows8"] == ["0:0", "1:0", "7:0", "0:1", "7:3", "8:0", "9:0", "19:3"]


def test_groups_of_columns_sweep_one_row_at_a_time(report):
    # the same grid in groups of 3 columns: tiles 0..2 are columns 0..2 of row 0
    assert report["cols3"] == ["0:0", "0:1", "2:1", "2:2", "10:1", "10:2", "11:0", "19:3"]


def test_split_tail_covers_every_tile_and_shortens_the_last_wave(report):
    """Tiles from split_tail_from on run as two 256 x 128 halves: every tile is covered once whole
    or by both halves, and the busiest pair's work never grows and shrinks whenever a tail splits
    (checked for 1..400 tiles over 1..100 pairs)."""
    assert report["split_failures"] == ["0"]


def test_split_tail_points_on_76_pairs(report):
    # 256 tiles (4096^2): 3 whole waves, the 28 left split into 56 halves; 80 tiles (4096 x 1280):
    # 4 left; 896 (a Llama MLP layer): 60 left, 120 halves would not fit one round, no split;
    # 400 (Qwen3-14B q/o): 20 left; 76 and 152: full waves; 40: one wave; 1360: 68 left, no split
    assert report["split_from"] == ["228", "76", "896", "380", "76", "40", "1360", "152"]
