"""The Newton-refined fp64 reciprocal and reciprocal square root the fp64
kernels use (finite_volume_shallow_gb300/csrc/swe_fastmath.cuh) stay within
2 units in the last place of CUDA's own 1.0 / x and rsqrt(x), over positive
arguments from 1e-300 to 1e300 and over the kernels' working range."""
import os
import subprocess

import pytest

from finite_volume_shallow_gb300 import build as B

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_fp64_reciprocals_within_two_ulp(tmp_path):
    exe = tmp_path / "fastmath_check"
    subprocess.run([B.nvcc(), *B.ARCH, "-O3", "-o", str(exe),
                    os.path.join(HERE, "cuda", "fastmath_check.cu")], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    status, ulp_rcp, ulp_rsq = out.stdout.split()
    assert status == "0", out.stdout   # cudaSuccess
    assert int(ulp_rcp) <= 2 and int(ulp_rsq) <= 2, out.stdout
