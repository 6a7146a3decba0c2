"""Every tcgen05 grouped-GEMM kernel on every call it can take: the one-SM
row-tile kernel alone (MOE_TC_KERNEL=1sm), and the weights-as-M kernel on SM
pairs with 128 (MOE_TC_KERNEL=sw) or 256 (MOE_TC_KERNEL=wide) weight rows
per CTA, each running the whole grouped-GEMM parity file (gathered rows
included) and the small whole-forward cases in a fresh process (the switch
is read once per process)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("kernel", ["1sm", "sw", "wide"])
def test_alternative_gemm_kernel_parity(kernel):
    env = dict(os.environ, MOE_TC_KERNEL=kernel)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_gpu_gemm.py"),
                        os.path.join(HERE, "test_gpu_ffn.py"), "-k",
                        "not full_size and not indexed", "-q", "-p", "no:cacheprovider"],
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
