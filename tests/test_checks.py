"""Rules of the checked build (host logic, no GPU).

Compiles tests/cuda/check_rules.cpp against the kernels' own checks.h with the
host C++ compiler and runs it: each predicate the checked build applies before
a TMA copy, a bulk copy or a TMEM access must accept exactly what its rule
allows.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_97_gb300", "csrc")


def test_check_rules(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "check_rules"
    subprocess.run([cxx, "-O2", "-std=c++17", "-Wall", "-Werror", "-I", CSRC,
                    os.path.join(ROOT, "tests", "cuda", "check_rules.cpp"), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    failed = [l for l in out.stdout.splitlines() if l.startswith("FAIL")]
    assert out.returncode == 0 and not failed, "\n".join(failed[:20])
    assert out.stdout.rstrip().endswith("ALL OK")
