"""The double-float helpers of the stochastic acceptance (csrc/common.cuh), compiled for the
host by nvcc and checked against exact fp64 arithmetic (tests/f2_host_check.cu): the sum and
the product of two floats reproduced exactly, sums of normalised pairs within 2^-44, the
order of fp64, the reciprocal within fp32 rounding. No GPU is used."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_double_float_helpers_against_fp64(tmp_path):
    from speculative_decoding_tree_parent_gb300 import build

    nvcc = build.nvcc()
    if not nvcc or not (os.path.exists(nvcc) or shutil.which(nvcc)):
        pytest.skip("nvcc not available")
    exe = tmp_path / "f2_host_check"
    subprocess.check_call([nvcc, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(ROOT, "speculative_decoding_tree_parent_gb300", "csrc"),
                           os.path.join(ROOT, "tests", "f2_host_check.cu"), "-o", str(exe)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout
    assert out.stdout.startswith("ok ")
