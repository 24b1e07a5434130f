"""The pool's plan cache reuses a plan only for exactly the metadata it was
built from (element-wise comparison of cu_q_lens, ctx_lens and q_positions and
of the planning parameters).  Host logic only: a small C++ program is
compiled against the library's planner and run here."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_attention_25_gb300", "csrc")


def test_plan_cache_key_is_exact(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "plan_cache_check")
    subprocess.run([cxx, "-O1", "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "native", "plan_cache_check.cpp"), os.path.join(CSRC, "plan.cpp"),
                    "-o", exe], check=True, capture_output=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout
