"""Block-scaled FP8 masked grouped GEMM (TileOPs "MoE Operators",
MoEGroupedGemmFP8FwdOp) on the tcgen05 kind::f8f6f4 path against the oracle,
with the pages' accuracy bound: on the valid rows |out - ref| <= atol + rtol
|ref|, atol = 2e-2 sqrt(max(1, K / 1024)), rtol = 2e-2.  Rows at or past a
count and everything after out stay unwritten; counts are clamped to
[0, max_m]."""
import math

import numpy as np
import pytest
import torch

from mixture_experts_ffn_gb300 import synth
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


def _codes(t):
    return t.view(torch.uint8).cpu().numpy()


def _check(got, ref, K, what):
    atol = 2e-2 * math.sqrt(max(1.0, K / 1024))
    err = np.abs(got - ref)
    bad = err > atol + 2e-2 * np.abs(ref)
    assert not bad.any(), (what, float(err.max()), int(bad.sum()))


@pytest.mark.parametrize("E,max_m,N,K,counts", [
    (3, 200, 256, 384, [-1, 150, 999]),     # clamped counts, max_m not a multiple of 128
    (2, 128, 128, 128, [128, 1]),           # one K block, a one-row expert
    (4, 300, 384, 256, None),               # three row tiles per expert
    (1, 64, 128, 1024, [64]),
    (5, 130, 256, 640, [0, 130, 129, 2, 77]),
    (4, 512, 512, 384, [300, 256, 257, 512]),  # two 256-row pair tiles per expert
    (3, 256, 640, 256, [129, 128, 255]),       # peer half with 0, 1 and 127 valid rows
    (1024, 2, 128, 128, None),                 # the most experts, one or two rows each
    (2, 1, 256, 384, [1, 0]),                  # one-row slab
])
def test_fp8_masked_gemm(moe, E, max_m, N, K, counts):
    inp = synth.make_fp8_masked(E, max_m, N, K, seed=E * 1000 + K, device="cuda", counts=counts)
    guard = 64
    flat = torch.full(((E * max_m + guard) * N,), float("nan"), dtype=torch.bfloat16,
                      device="cuda")
    out = flat[: E * max_m * N].view(E, max_m, N)
    moe.moe_grouped_gemm_fp8_masked(inp["a"], inp["a_scale"], inp["b"], inp["b_scale"],
                                    inp["counts"], out=out)
    again = moe.moe_grouped_gemm_fp8_masked(inp["a"], inp["a_scale"], inp["b"], inp["b_scale"],
                                            inp["counts"])
    torch.cuda.synchronize()
    ref = O.grouped_gemm_fp8_masked(_codes(inp["a"]), inp["a_scale"].cpu().numpy(),
                                    _codes(inp["b"]), inp["b_scale"].cpu().numpy(),
                                    inp["counts"].cpu().numpy(), dtype=None)
    got = out.float().cpu().numpy()
    for g in range(E):
        m = min(max(int(inp["counts"][g]), 0), max_m)
        _check(got[g, :m], ref[g, :m], K, f"expert {g}")
        assert np.isnan(got[g, m:]).all(), "rows past the count were written"
        assert torch.equal(out[g, :m], again[g, :m]), "not deterministic"
    assert torch.isnan(flat[E * max_m * N:]).all(), "wrote past out"


def test_fp8_masked_gemm_deepseek_size_sampled(moe):
    """DeepSeek-V3-style expert-parallel shapes (8 local experts, up to 256
    rows each, N 4096, K 7168); the oracle checks six rows of every expert,
    from both 128-row halves of its tile, the last valid row included."""
    E, max_m, N, K = 8, 256, 4096, 7168
    inp = synth.make_fp8_masked(E, max_m, N, K, seed=3, device="cuda")
    out = moe.moe_grouped_gemm_fp8_masked(inp["a"], inp["a_scale"], inp["b"], inp["b_scale"],
                                          inp["counts"])
    torch.cuda.synchronize()
    counts = inp["counts"].cpu().numpy()
    for g in range(E):
        c = int(min(max(counts[g], 0), max_m))
        rows = sorted({r for r in (0, 1, 77, 127, 128, c - 1) if 0 <= r < c})
        ref = O.grouped_gemm_fp8_masked(_codes(inp["a"][g:g + 1, rows]),
                                        inp["a_scale"][g:g + 1, rows].cpu().numpy(),
                                        _codes(inp["b"][g:g + 1]),
                                        inp["b_scale"][g:g + 1].cpu().numpy(), [len(rows)],
                                        dtype=None)
        _check(out[g:g + 1, rows].float().cpu().numpy(), ref, K, f"DeepSeek-V3 size, expert {g}")


def test_fp8_masked_gemm_rejects(moe):
    inp = synth.make_fp8_masked(2, 128, 128, 256, seed=9, device="cuda")
    with pytest.raises(moe.MoEError) as ei:  # K not a multiple of 128
        moe.moe_grouped_gemm_fp8_masked(inp["a"][:, :, :200].contiguous(), inp["a_scale"],
                                        inp["b"][:, :, :200].contiguous(), inp["b_scale"],
                                        inp["counts"])
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
