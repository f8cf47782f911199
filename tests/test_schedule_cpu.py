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
