"""The decode copy plans, built and checked on the host for many shapes and
grid sizes, without a GPU:
- the one-shot kernel's (csrc/decode_oneshot.h) by tests/plan_check.cu:
  16-byte alignment and bounds of every bulk copy, the bytes each barrier
  expects, and that every code and scale byte the kernel reads was copied
  from the right record;
- the ring kernel's chunk plan (csrc/decode_ring_plan.h) by
  tests/ring_plan_check.cu: every row covered exactly once, slot capacity,
  copy alignment, and the scale bytes the consumers read."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    pytest.skip("nvcc not found")


def test_decode_plan_on_host(tmp_path):
    exe = tmp_path / "plan_check"
    cmd = [_nvcc(), "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "block_scaled_fp4_softmax_gb300", "csrc"),
           "-o", str(exe), os.path.join(HERE, "plan_check.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=900)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-3000:]
    assert ", 0 failed" in r.stdout


def test_ring_plan_on_host(tmp_path):
    exe = tmp_path / "ring_plan_check"
    cmd = [_nvcc(), "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "block_scaled_fp4_softmax_gb300", "csrc"),
           "-o", str(exe), os.path.join(HERE, "ring_plan_check.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=900)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-3000:]
    assert ", 0 failed" in r.stdout

