"""Launch plans checked on the host: the tree-growth kernel's staging depth
and shared-memory size for every shape the interface admits (the plan
functions of sv_grow.cuh, compiled with nvcc into a host program)."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_verification_56_gb300", "csrc")


def test_grow_plan_fits_every_admitted_shape(tmp_path):
    from speculative_decoding_verification_56_gb300 import build
    try:
        nvcc = build._nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    exe = tmp_path / "grow_plan_check"
    cmd = [nvcc, *build.ARCH_FLAGS, "-std=c++17", "-O1", "-I", build.INCLUDE, "-I", CSRC,
           os.path.join(ROOT, "tests", "grow_plan_check.cu"), "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-2000:]
    assert "shapes checked" in r.stdout
