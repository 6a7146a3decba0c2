"""The two-SM (cta_group::2) variant of the tcgen05 grouped GEMM, selected with
MOE_TC_2SM=1, runs the whole grouped-GEMM parity file in a fresh process (the
switch is read once per process)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_two_sm_gemm_parity():
    env = dict(os.environ, MOE_TC_2SM="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_gpu_gemm.py"),
                        "-q", "-p", "no:cacheprovider"], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
