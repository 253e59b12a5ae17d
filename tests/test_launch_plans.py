"""Host-side checks of the CUDA sources, no GPU needed: the tree-growth
kernel's staging depth and shared-memory size for every shape the interface
admits (the plan functions of sv_grow.cuh, compiled with nvcc into a host
program), the fused LM head's plan for every row-group size (sv_lmhead.cuh,
likewise), and the provenance of the FMA-pipe 2^x coefficients."""
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


def test_lmhead_plan_fits_every_row_group(tmp_path):
    from speculative_decoding_verification_56_gb300 import build
    try:
        nvcc = build._nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    exe = tmp_path / "lmhead_plan_check"
    cmd = [nvcc, *build.ARCH_FLAGS, "-std=c++17", "-O1", "-I", build.INCLUDE, "-I", CSRC,
           os.path.join(ROOT, "tests", "lmhead_plan_check.cu"), "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-2000:]
    assert "6 row-group sizes checked" in r.stdout


def test_exp2_polynomial_comes_from_the_committed_fit():
    # the FMA-pipe 2^x in sv_device.cuh uses the coefficients that
    # csrc/fit_exp2_poly.py (Cody-Waite reduction, Remez exchange) prints
    import re
    import sys
    script = os.path.join(CSRC, "fit_exp2_poly.py")
    r = subprocess.run([sys.executable, script], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    fitted = [float(m) for m in re.findall(r"c\d = ([0-9.eE+-]+)", r.stdout)]
    assert len(fitted) == 6
    src = open(os.path.join(CSRC, "sv_device.cuh")).read()
    body = src[src.index("float exp2_fma(float x)"):]
    body = body[:body.index("\n}\n")]
    used = [float(m) for m in re.findall(r"([0-9][0-9.]*e?-?[0-9]*)f", body)
            if "." in m]
    # the Horner chain lists c5 first and c0 last
    coeffs = [c for c in used if c not in (12582912.0, 126.0)]
    assert coeffs[::-1] == fitted, (coeffs, fitted)
