"""libfattn used from plain C (tests/c_abi/fa_c_example.c): the program
compiles against include/fattn.h and links against libfattn.so and the CUDA
runtime alone (CPU test); on the GPU it runs the forward and the
deterministic backward on buffers it allocates itself, and its outputs match
the oracle (GPU test).  A second program (tests/c_abi/fa_c_reset.c) runs the
forward and the no-allocation backward, resets the device, and runs them
again: what the library set up once per device must be set up again in the
new context, and the outputs must be identical."""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import parity_util as U
from exact_attention_93_gb300 import build, fattn, workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "c_abi", "fa_c_example.c")
RESET_SRC = os.path.join(HERE, "c_abi", "fa_c_reset.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_example(out_dir, src=SRC, name="fa_c_example"):
    build.build()
    exe = os.path.join(out_dir, name)
    lib_dir = os.path.dirname(fattn.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", src,
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                    "-L", lib_dir, "-lfattn", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}",
                    "-lm", "-o", exe], check=True)
    return exe


def test_example_compiles_and_links(tmp_path):
    assert os.path.exists(compile_example(str(tmp_path)))
    assert os.path.exists(compile_example(str(tmp_path), RESET_SRC, "fa_c_reset"))


@pytest.mark.gpu
def test_outputs_identical_across_a_device_reset(tmp_path):
    exe = compile_example(str(tmp_path), RESET_SRC, "fa_c_reset")
    r = subprocess.run([exe, "1", "2", "300", "64", "1"], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_example_matches_oracle(tmp_path):
    exe = compile_example(str(tmp_path))
    w = W.custom(1, 2, 200, 64, "bf16", causal=True, seed=51)
    inputs = W.make_inputs(w)
    raw = b"".join(inputs[n].contiguous().view(torch.int16).numpy().tobytes()
                   for n in ("q", "k", "v", "do"))
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    fin.write_bytes(raw)
    r = subprocess.run([exe, str(fin), str(fout), str(w.B), str(w.H), str(w.N), str(w.D), "1"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    n, rows = w.B * w.H * w.N * w.D, w.B * w.H * w.N
    buf = fout.read_bytes()

    def bf16_at(off):
        h = np.frombuffer(buf, dtype=np.uint16, count=n, offset=off).astype(np.uint32) << 16
        return h.view(np.float32).astype(np.float64).reshape(w.B, w.H, w.N, w.D)

    o = bf16_at(0)
    lse = np.frombuffer(buf, dtype=np.float32, count=rows, offset=2 * n).reshape(w.B, w.H, w.N)
    dq, dk, dv = (bf16_at(2 * n + 4 * rows + i * 2 * n) for i in range(3))
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], w.scale, True,
                           dout=inputs["do"])
    assert U.o_err(o, ref["o"], "bf16") <= U.TOL_O
    assert U.max_abs(lse, ref["lse"]) <= U.TOL_LSE
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert U.rel_err(got, ref[name]) <= U.TOL_GRAD_REL, name
