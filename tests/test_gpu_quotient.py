"""The pack kernel's codecs take rn(x / s) from Markstein's correction
z = fma(fma(-y, s, x), r, y), r = rn(1/s), y = rn(x r), instead of an IEEE
divide.  This compiles tests/cuda/quotient_check.cu and compares z with CUDA's
__fdiv_rn for every pair of binary32 significands (x, s in [1, 2): 2^46
pairs, about 40 s on a GB300), after the bf16 and fp16 significand grids."""
import os
import re
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "cuda", "quotient_check.cu")


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path_factory.mktemp("quotient") / "quotient_check")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe, SRC],
                   check=True)
    return exe


@pytest.mark.parametrize("x_bits", [7, 10, 23], ids=["bf16", "fp16", "binary32"])
def test_corrected_quotient_equals_ieee_division(checker, x_bits):
    out = subprocess.run([checker, str(x_bits)], capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stdout + out.stderr
    m = re.search(r"pairs (\d+) mismatches (\d+)", out.stdout)
    assert m, out.stdout
    assert int(m.group(1)) == (1 << x_bits) << 23
    assert int(m.group(2)) == 0, out.stdout
