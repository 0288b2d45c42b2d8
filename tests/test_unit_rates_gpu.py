"""Measured per-SM rates of the instructions the elementwise steps use.

The benchmark's exponential-rate ceiling takes ex2.approx.ftz.f32 at 32
lanes per clock per SM, and the kernels' notes quote the e4m3 and bf16 pair
conversions' rates, the half-precision exponential's and conversions' rates
(the alternatives for the 8-bit softmax) and the cycles per tensor-core
product of each shape the tile kernels issue; these tests measure them on
the GPU (standalone programs under tests/rates/, compiled here for sm_103a)
and print them.
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
MMA_SRC = os.path.join(HERE, "rates", "mma_rates.cu")
CSRC = os.path.join(os.path.dirname(HERE), "exact_attention_93_gb300", "csrc")

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
    assert r["ex2_approx_f16x2_instr_per_clk_sm"] > 0 and r["cvt_f32_f16_per_clk_sm"] > 0
    assert r["ex2_f32_with_cvt_f16x2_f32_instr_per_clk_sm"] > 0


def test_tensor_core_product_rates():
    """Cycles per bf16 tcgen05.mma product, all SMs at once: M128 N128 K16
    and M128 N256 K16 near their full rates (64 and 128 cycles), M128 N64 K16
    with both operands in shared memory slower than half the N128 product
    (6 KB of operands per product at the shared-memory port's 128 bytes per
    cycle), A from TMEM as fast as from shared memory."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "mma_rates")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I" + CSRC, "-o", exe, MMA_SRC], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=120)
    r = json.loads(out.stdout.strip().splitlines()[-1])
    print(f"[rates] {r}")
    assert 0.9 * 64 <= r["m128n128k16_ss"] <= 1.5 * 64
    assert 0.9 * 128 <= r["m128n256k16_ss"] <= 1.5 * 128
    assert r["m128n64k16_ss"] >= 0.9 * 32 and r["m128n64k16_ss"] > 0.55 * r["m128n128k16_ss"]
    assert r["m128n128k16_ts"] <= 1.5 * 64
