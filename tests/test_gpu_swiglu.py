"""Standalone SwiGLU op against the oracle and the golden points."""
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

from gpu_cases import np_
from tolerances import assert_rounded_once

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("with_up,fusion", [(True, 2), (False, 1), (False, 2)])
@pytest.mark.parametrize("limit,alpha,beta", [(7.0, 1.702, 1.0), (0.0, 1.0, 0.0), (-1.0, 0.5, 2.0),
                                              (2.5, 3.0, -0.5)])
@pytest.mark.parametrize("R,I", [(257, 96),    # 16-byte items
                                 (33, 97),     # odd width: one element per thread
                                 (300, 2880)])  # gpt-oss-style intermediate width
def test_swiglu(moe, dtype, with_up, fusion, limit, alpha, beta, R, I):
    g = torch.Generator().manual_seed(11)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    gate = (torch.randn((R, I if with_up else 2 * I), generator=g) * 6).to(tdt)
    up = (torch.randn((R, I), generator=g) * 6).to(tdt) if with_up else None
    out = moe.swiglu(gate.cuda(), None if up is None else up.cuda(), fusion, limit, alpha, beta)
    torch.cuda.synchronize()
    exact = O.swiglu_op(np_(gate), None if up is None else np_(up), I, fusion, limit, alpha, beta,
                        None)
    assert_rounded_once(np_(out), exact, dtype, "swiglu")


def test_swiglu_golden_points_on_gpu(moe):
    path = os.path.join(os.path.dirname(__file__), "golden", "swiglu_points.txt")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        gv, lv, limit, alpha, beta, expected = [float(v) for v in line.split("#")[0].split()]
        gate = torch.tensor([[gv]], dtype=torch.float32, device="cuda")
        up = torch.tensor([[lv]], dtype=torch.float32, device="cuda")
        out = moe.swiglu(gate, up, 2, limit, alpha, beta)
        assert float(out[0, 0]) == pytest.approx(expected, rel=2e-6, abs=1e-7), line
