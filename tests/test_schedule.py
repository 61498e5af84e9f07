"""The Newton-Schulz tile planner on the host: every list covers its phase's tiles once,
the persistent launch's per-iteration lists cannot deadlock under the kernel's waiting
rules, and they beat per-phase lists in matrix order on the planner's cost model.  The
checks are in schedule_check.cpp, built here with g++ against the planner's source."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "muon_optimizer_step_gb300", "csrc")


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_tile_planner(tmp_path):
    exe = str(tmp_path / "schedule_check")
    subprocess.run(["g++", "-std=c++17", "-O2", "-I", CSRC,
                    os.path.join(ROOT, "tests", "schedule_check.cpp"),
                    os.path.join(CSRC, "layout.cpp"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout + r.stderr
