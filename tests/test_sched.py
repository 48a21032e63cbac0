"""Static work schedule of the persistent kernels (host logic, no GPU).

Compiles tests/cuda/sched_check.cpp against the kernels' own schedule header
with the host C++ compiler and runs it: every (tile, head) item must go to
exactly one CTA for every mode, shape and grid size tried, and the mode the
host picks must balance the causal tile costs on the large shapes.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_97_gb300", "csrc")


def test_schedule_covers_every_item_once(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "sched_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(ROOT, "tests", "cuda", "sched_check.cpp"), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    failed = [l for l in out.stdout.splitlines() if l.startswith("FAIL")]
    assert out.returncode == 0 and not failed, "\n".join(failed[:20])
    assert out.stdout.rstrip().endswith("ALL OK")
