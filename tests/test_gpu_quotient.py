"""The block quotient of the quantising kernels (Markstein's correction from
the block's correctly rounded reciprocal, csrc/quotient.cuh) gives the same
e4m3 codes as CUDA's IEEE division for every input the act_quant rule can
produce: every finite bf16 amax, its scale in both formats, every bf16 x with
|x| <= amax (about 1.07e9 pairs per format). The checker is compiled from
tests/cuda/quotient_check.cu around the library's own header."""
import os
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "fp8_block_scaled_quant_gb300", "csrc")


def test_block_quotient_codes_equal_ieee_division_exhaustively():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "quotient_check")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-I", CSRC, "-o", exe,
                        os.path.join(HERE, "cuda", "quotient_check.cu")], check=True, capture_output=True, timeout=300)
        res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    lines = res.stdout.strip().splitlines()
    assert res.returncode == 0, res.stdout + res.stderr
    assert len(lines) == 2 and all(" mismatches 0" in ln for ln in lines), res.stdout
    assert all(int(ln.split()[2]) > 10 ** 9 for ln in lines), res.stdout
