"""The tensor-core rates behind the attention consumer's precision choice,
measured on this GPU (tests/cuda/mma_rate.cu: back-to-back tcgen05.mma from
shared memory into TMEM, one CTA per SM, CUDA events).  The consumer widens
INT8 Q/K and E4M3 V to fp16 and runs kind::f16; kind::i8 has no form for
sm_103a (ptxas rejects it), and kind::f8f6f4 with E4M3 operands is measured
beside kind::f16 here.  Checks only that the rates are positive and in the
nominal range of the part (the figures go to the design doc by hand)."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cuda", "mma_rate.cu")
CSRC = os.path.join(os.path.dirname(HERE), "quantize_pack_gb300", "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")


def test_tensor_core_rates(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "mma_rate")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", CSRC, "-I", INCLUDE, SRC, "-o", exe], check=True)
    out = subprocess.run([exe, "20000"], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    rates = {}
    for line in out.stdout.strip().splitlines():
        kind, M, N, K, iters, ms, tflops = line.split()
        rates[(kind, int(N))] = float(tflops)
        print(line)
    assert set(rates) == {("f16", 128), ("f16", 256), ("f8f6f4_e4m3", 128), ("f8f6f4_e4m3", 256)}
    for (kind, N), r in rates.items():
        nominal = 2250.0 if kind == "f16" else 4500.0
        assert 0.2 * nominal < r < 1.2 * nominal, (kind, N, r)
