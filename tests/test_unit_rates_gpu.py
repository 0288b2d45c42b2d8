"""Measured per-SM rates of the instructions the elementwise steps use.

The benchmark's exponential-rate ceiling takes ex2.approx.ftz.f32 at 32
lanes per clock per SM, and the kernels' notes quote the e4m3 and bf16 pair
conversions' rates; this test measures them on the GPU (a standalone program,
tests/rates/unit_rates.cu, compiled here for sm_103a) and prints them.
"""
import json
import os
import shutil
import subprocess
import sys
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rates", "unit_rates.cu")

sys.path.insert(0, os.path.dirname(HERE))
import bench  # noqa: E402  (the constant this test stands behind)


def test_special_function_rates():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "unit_rates")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-o", exe, SRC], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=120)
    r = json.loads(out.stdout.strip().splitlines()[-1])
    print(f"[rates] {r}")
    # the constant the benchmark's exponential ceiling uses
    assert abs(r["ex2_approx_f32_per_clk_sm"] - bench.EX2_PER_CLK_SM) <= 0.1 * bench.EX2_PER_CLK_SM
    assert r["cvt_e4m3x2_f32_instr_per_clk_sm"] > 0 and r["cvt_bf16x2_f32_instr_per_clk_sm"] > 0
