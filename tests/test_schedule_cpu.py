"""The stream-K schedule the split kernels run (paged_kv_cache_209_gb300/csrc/
pkv_schedule.cuh), compiled for the host and checked against brute force by
tests/schedule_check.cu: the cost-weighted CTA split of the decode kernels
(range starts, the CTA of a unit, the pieces of every segment and their
CTAs), the equal split of the multi-query kernels, and the walker that turns
a CTA's range into segment pieces. No GPU needed: nvcc compiles host code."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_schedule_against_brute_force(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "schedule_check")
    src = os.path.join(ROOT, "tests", "schedule_check.cu")
    inc = os.path.join(ROOT, "paged_kv_cache_209_gb300", "csrc")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", inc, src, "-o", exe], check=True, capture_output=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok "), r.stdout
