"""Grouped GEMMs (gate_up + fused activation, and down) against the oracle on
ragged expert segments: empty experts, segments shorter and longer than a
128-row tile, column tiles and k-blocks with ragged tails, every activation
layout, with and without bias, on the tcgen05 path, the SIMT path and fp32."""
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

from gpu_cases import LazyExperts, np_
from tolerances import assert_rounded_once

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


def _problem(counts, Hk, N1, dtype, bias, seed):
    g = torch.Generator().manual_seed(seed)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    E = len(counts)
    M = int(sum(counts))
    a = torch.randn((M, Hk), generator=g).to(tdt)
    w = (torch.randn((E, N1, Hk), generator=g) / Hk ** 0.5).to(tdt)
    b = (torch.randn((E, N1), generator=g) * 0.02).to(tdt) if bias else None
    seg_end = torch.tensor(np.cumsum(counts), dtype=torch.int32)
    return a, w, b, seg_end


ACTS = {
    "silu": dict(kind=0, swiglu_fusion=2),
    "swiglu_inter": dict(kind=1, swiglu_fusion=1, limit=7.0, alpha=1.702, beta=1.0),
    "swiglu_concat": dict(kind=1, swiglu_fusion=2, limit=3.0, alpha=1.0, beta=0.0),
    "swiglu_noclamp": dict(kind=1, swiglu_fusion=1, limit=0.0, alpha=1.3, beta=0.5),
    "identity": dict(kind=2),
    "gelu_mul": dict(kind=3),
    "relu": dict(kind=4),
    "gelu": dict(kind=5),
    "silu_plain": dict(kind=6),
}
GATED = (0, 1, 3)


@pytest.mark.parametrize("counts,Hk,F,act,bias,dtype,simt", [
    ([3, 0, 130, 1, 300], 256, 192, "silu", False, "bf16", False),
    ([129, 127, 0, 256], 320, 160, "swiglu_inter", True, "bf16", False),
    ([129, 127, 0, 256], 320, 160, "swiglu_concat", True, "bf16", False),
    ([50, 0, 0, 77, 200], 200, 96, "swiglu_noclamp", False, "bf16", False),  # ragged k-block
    ([200, 56, 100], 128, 384, "identity", True, "bf16", False),
    ([1], 64, 8, "silu", False, "bf16", False),                              # one row
    ([0, 0, 0, 5], 64, 128, "silu", True, "bf16", False),                    # leading empty experts
    ([3, 0, 130, 1, 300], 256, 192, "silu", True, "bf16", True),             # SIMT, bf16
    ([129, 127, 0, 256], 320, 160, "swiglu_inter", True, "bf16", True),
    ([16] * 8, 128, 64, "silu", False, "f32", False),                        # fp32 (SIMT)
    ([40, 0, 25, 63], 100, 50, "swiglu_inter", True, "f32", False),
    ([300, 5, 0, 211], 132, 36, "silu", False, "bf16", False),               # F % 8 != 0 -> SIMT
    ([3, 0, 130, 1, 300], 256, 192, "gelu_mul", True, "bf16", False),       # gelu_and_mul
    ([129, 127, 0, 256], 320, 160, "gelu_mul", False, "bf16", True),
    ([40, 0, 25, 63], 100, 48, "gelu_mul", True, "f32", False),
    ([200, 56, 100], 128, 384, "relu", True, "bf16", False),                 # non-gated
    ([200, 56, 100], 128, 384, "gelu", False, "bf16", False),
    ([129, 1, 300], 256, 256, "silu_plain", True, "bf16", False),
    ([40, 0, 25, 63], 100, 48, "gelu", True, "f32", False),
    ([40, 0, 25, 63], 100, 44, "silu_plain", False, "bf16", True),
])
def test_gemm_act(moe, counts, Hk, F, act, bias, dtype, simt):
    spec = ACTS[act]
    N1 = 2 * F if spec["kind"] in GATED else F
    a, w, b, seg_end = _problem(counts, Hk, N1, dtype, bias, seed=len(counts) * 1000 + Hk)
    M = a.shape[0]
    p = moe.act_params(**spec)
    out = torch.full((M + 7, F), float("nan"), dtype=a.dtype, device="cuda")  # + unwritten rows
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    old = moe.moe_set_gemm_simt(simt)
    try:
        a_pad = torch.cat([a, torch.zeros((7, Hk), dtype=a.dtype)])  # rows outside every segment
        moe.moe_grouped_gemm_act(a_pad.cuda(), w.cuda(),
                                 seg_end.cuda(), F, p, None if b is None else b.cuda(),
                                 out=out, ws=ws)
        assert moe.moe_sync_status(ws) == moe.MOE_OK
    finally:
        moe.moe_set_gemm_simt(old)
    exact = O.grouped_gemm_act(np_(a), np_(w), np_(seg_end), F, spec["kind"],
                               spec.get("swiglu_fusion", 2), spec.get("limit", 0.0),
                               spec.get("alpha", 1.0), spec.get("beta", 0.0),
                               None if b is None else np_(b), dtype=None)
    got = np_(out)
    assert np.isnan(got[M:]).all(), "rows past the last segment were written"
    assert_rounded_once(got[:M], exact, dtype, f"gemm_act {act}")


@pytest.mark.parametrize("simt", [False, True])
def test_gemm_act_largest_expert_count(moe, simt):
    """E = 1024 (the largest accepted): mostly empty or one-row segments, a few
    longer ones, so the shared tile builder's scan runs over every expert."""
    rng = np.random.default_rng(1024)
    counts = rng.choice([0, 0, 1, 2, 5, 130], size=1024).tolist()
    a, w, b, seg_end = _problem(counts, 64, 128, "bf16", True, seed=1024)
    M, F = a.shape[0], 64
    out = torch.full((M, F), float("nan"), dtype=a.dtype, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    old = moe.moe_set_gemm_simt(simt)
    try:
        moe.moe_grouped_gemm_act(a.cuda(), w.cuda(), seg_end.cuda(), F, moe.act_params(kind=0),
                                 b.cuda(), out=out, ws=ws)
        assert moe.moe_sync_status(ws) == moe.MOE_OK
    finally:
        moe.moe_set_gemm_simt(old)
    exact = O.grouped_gemm_act(np_(a), np_(w), np_(seg_end), F, 0, 2, 0.0, 1.0, 0.0, np_(b),
                               dtype=None)
    assert_rounded_once(np_(out), exact, "bf16", "gemm_act E=1024")


@pytest.mark.parametrize("counts,F,H,bias,dtype,simt", [
    ([3, 0, 130, 1, 300], 192, 320, True, "bf16", False),
    ([257, 0, 31], 128, 256, False, "bf16", False),
    ([10, 20, 0, 400], 72, 136, True, "bf16", False),      # ragged k-block (72 = 64 + 8)
    ([3, 0, 130, 1, 300], 192, 320, True, "bf16", True),
    ([16] * 8, 64, 128, False, "f32", False),
])
def test_gemm_down(moe, counts, F, H, bias, dtype, simt):
    a, w, b, seg_end = _problem(counts, F, H, dtype, bias, seed=7 + F)
    M = a.shape[0]
    out = torch.full((M, H), float("nan"), dtype=a.dtype, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    old = moe.moe_set_gemm_simt(simt)
    try:
        moe.moe_grouped_gemm_down(a.cuda(), w.cuda(), seg_end.cuda(),
                                  None if b is None else b.cuda(), out=out, ws=ws)
        assert moe.moe_sync_status(ws) == moe.MOE_OK
    finally:
        moe.moe_set_gemm_simt(old)
    exact = O.grouped_gemm_down(np_(a), np_(w), np_(seg_end), None if b is None else np_(b),
                                dtype=None)
    assert_rounded_once(np_(out), exact, dtype, "gemm_down")


def test_gemm_act_large_sampled(moe):
    """Qwen3-style shapes (32768 rows over 128 experts, H 2048, F 768) on the
    tcgen05 path; the oracle checks the rows of four experts and 64 random rows."""
    g = torch.Generator().manual_seed(5)
    E, Hk, F = 128, 2048, 768
    counts = torch.multinomial(torch.ones(E), 32768, replacement=True, generator=g)
    counts = torch.bincount(counts, minlength=E).numpy()
    a = torch.randn((32768, Hk), generator=g).to(torch.bfloat16).cuda()
    gw = torch.Generator(device="cuda").manual_seed(6)
    w = (torch.randn((E, 2 * F, Hk), generator=gw, device="cuda") / Hk ** 0.5).to(torch.bfloat16)
    seg_end = torch.tensor(np.cumsum(counts), dtype=torch.int32, device="cuda")
    out = moe.moe_grouped_gemm_act(a, w, seg_end, F, moe.act_params(0))
    torch.cuda.synchronize()
    ends = np.cumsum(counts)
    starts = ends - counts
    rows = set()
    for e in (0, 1, 77, 127):
        rows.update(range(starts[e], ends[e]))
    rows.update(np.random.default_rng(0).integers(0, 32768, 64).tolist())
    rows = np.array(sorted(rows))
    exp_of_row = np.searchsorted(ends, rows, side="right")
    sub_counts = np.bincount(exp_of_row, minlength=E)
    a_np = a[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    exact = O.grouped_gemm_act(a_np, LazyExperts(w), np.cumsum(sub_counts), F, 0, dtype=None)
    assert_rounded_once(np_(out)[rows], exact, "bf16", "gemm_act large")


@pytest.mark.parametrize("T,K,E,H,F,act,bias", [
    (64, 2, 5, 256, 192, "silu", False),
    (300, 4, 7, 320, 160, "swiglu_inter", True),
    (300, 4, 7, 320, 160, "swiglu_concat", True),
    (97, 8, 16, 128, 64, "silu", True),      # ragged segments, some experts empty
    (1, 1, 3, 64, 8, "silu", False),         # one route
    (513, 2, 4, 200, 96, "swiglu_noclamp", False),  # long segments, ragged k-block
    (300, 4, 7, 256, 128, "gelu_mul", True),
    (1200, 2, 4, 256, 128, "silu", True),    # ~600-row segments: several 256-row tiles
])
def test_gemm_act_gathered(moe, T, K, E, H, F, act, bias):
    """The gate_up GEMM reading its rows through row_to_route from the
    token-ordered hidden states equals the GEMM on the permuted copy bit for
    bit, and the oracle on the rows the oracle's own permutation selects."""
    assert K <= E, "top-k ids are distinct experts"
    spec = ACTS[act]
    N1 = 2 * F
    g = torch.Generator().manual_seed(T * 31 + H)
    hidden = torch.randn((T, H), generator=g).to(torch.bfloat16)
    w = (torch.randn((E, N1, H), generator=g) / H ** 0.5).to(torch.bfloat16)
    b = (torch.randn((E, N1), generator=g) * 0.02).to(torch.bfloat16) if bias else None
    ids = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).to(torch.int32)
    p = moe.act_params(**spec)
    perm = moe.moe_permute(ids.cuda(), E, hidden.cuda())
    bc = None if b is None else b.cuda()
    got = moe.moe_grouped_gemm_act_gathered(hidden.cuda(), perm["row_to_route"], K, w.cuda(),
                                            perm["seg_end"], F, p, bc)
    ref_perm = moe.moe_grouped_gemm_act(perm["expert_input"], w.cuda(), perm["seg_end"], F, p, bc)
    torch.cuda.synchronize()
    assert torch.equal(got, ref_perm), "gathered rows differ from the permuted-copy GEMM"
    o = O.permute(ids.numpy(), E)
    assert np.array_equal(np_(perm["row_to_route"]).astype(np.int32), o["row_to_route"])
    a = O.gather_rows(np_(hidden), o["row_to_route"], K)
    exact = O.grouped_gemm_act(a, np_(w), o["seg_end"], F, spec["kind"],
                               spec.get("swiglu_fusion", 2), spec.get("limit", 0.0),
                               spec.get("alpha", 1.0), spec.get("beta", 0.0),
                               None if b is None else np_(b), dtype=None)
    assert_rounded_once(np_(got), exact, "bf16", f"gemm_act_gathered {act}")


def test_gemm_act_gathered_rejects_unsupported(moe):
    """fp32 (no tensor-core path) is refused, not silently computed elsewhere."""
    hidden = torch.randn((8, 64), device="cuda")
    w = torch.randn((2, 16, 64), device="cuda")
    seg_end = torch.tensor([8, 16], dtype=torch.int32, device="cuda")
    r2r = torch.arange(16, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_grouped_gemm_act_gathered(hidden, r2r, 2, w, seg_end, 8, moe.act_params(0))
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("layout,counts,max_m,K,F,act,bias,dtype", [
    ("per_row", [3, 0, 130, 1, 300], 0, 256, 192, "silu", True, "bf16"),
    ("per_row", [200, 56, 100], 0, 128, 384, None, True, "bf16"),
    ("per_row", [16] * 8, 0, 128, 64, "gelu", False, "f32"),
    ("masked", [130, -2, 99999, 7], 200, 256, 128, "gelu_mul", True, "bf16"),  # clamped counts
    ("masked", [50, 0, 200], 200, 128, 256, None, True, "bf16"),
    ("masked", [5, 3], 8, 64, 32, "relu", False, "f32"),
])
def test_gemm_row_layouts(moe, layout, counts, max_m, K, F, act, bias, dtype):
    """MoEGroupedGemmFwdOp's per_row and masked layouts: against the oracle on
    the valid rows, untouched rows past the masked counts, and bit for bit the
    segment-end result on the same rows."""
    spec = ACTS[act] if act else None
    N1 = 2 * F if spec and spec["kind"] in GATED else F
    E = len(counts)
    eff = [min(max(c, 0), max_m) for c in counts] if layout == "masked" else counts
    a, w, b, seg_end = _problem(eff, K, N1, dtype, bias, seed=K * 10 + E)
    p = moe.act_params(**spec) if spec else None
    tdt = a.dtype
    if layout == "per_row":
        ids = torch.repeat_interleave(torch.arange(E), torch.tensor(counts)).to(torch.int32)
        got = moe.moe_grouped_gemm(a.cuda(), w.cuda(), moe.MOE_LAYOUT_PER_ROW, ids.cuda(), F, p,
                                   None if b is None else b.cuda())
        meta, a_in = ids.numpy(), np_(a)
    else:
        slab = torch.zeros((E, max_m, K), dtype=tdt)
        pos = 0
        for e, m in enumerate(eff):
            slab[e, :m] = a[pos:pos + m]
            pos += m
        out = torch.full((E, max_m, F), float("nan"), dtype=tdt, device="cuda")
        got = moe.moe_grouped_gemm(slab.cuda(), w.cuda(), moe.MOE_LAYOUT_MASKED,
                                   torch.tensor(counts, dtype=torch.int32).cuda(), F, p,
                                   None if b is None else b.cuda(), out=out)
        meta, a_in = np.array(counts), np_(slab)
    torch.cuda.synchronize()
    kw = dict(act=spec["kind"], F=F, fusion=spec.get("swiglu_fusion", 2), limit=spec.get("limit", 0.0),
              alpha=spec.get("alpha", 1.0), beta=spec.get("beta", 0.0)) if spec else {}
    exact = O.grouped_gemm_layout(a_in, np_(w), layout, meta, bias=None if b is None else np_(b),
                                  dtype=None, **kw)
    g = np_(got)
    if layout == "masked":
        for e, m in enumerate(eff):
            assert np.isnan(g[e, m:]).all(), "rows past the count were written"
        g = np.concatenate([g[e, :m] for e, m in enumerate(eff)])
        exact = np.concatenate([exact[e, :m] for e, m in enumerate(eff)])
    assert_rounded_once(g, exact, dtype, f"{layout} {act}")
    # the same rows through the segment-end layout, bit for bit
    if spec:
        ref = moe.moe_grouped_gemm_act(a.cuda(), w.cuda(), seg_end.cuda(), F, p,
                                       None if b is None else b.cuda())
    else:
        ref = moe.moe_grouped_gemm_down(a.cuda(), w.cuda(), seg_end.cuda(),
                                        None if b is None else b.cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g, np_(ref))


def test_pair_kernel_workspace_reuse(moe):
    """The SM-pair kernel (K >= 2048, segments averaging >= 128 rows) hands
    out the tiles of its last rounds from a counter in the workspace's status
    area, which the launch's last pair resets.  Consecutive calls of
    different shapes on one workspace give bit for bit the results of fresh
    workspaces, match the oracle, and leave the counters at zero."""
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    cases = [([300, 0, 200, 100], 2048, 128, "silu"), ([129, 640, 7, 0, 260], 2304, 192, "silu"),
             ([300, 0, 200, 100], 2048, 128, "swiglu_inter")]
    for i, (counts, Hk, F, act) in enumerate(cases):
        spec = ACTS[act]
        a, w, b, seg_end = _problem(counts, Hk, 2 * F, "bf16", True, seed=40 + i)
        args = (a.cuda(), w.cuda(), seg_end.cuda(), F, moe.act_params(**spec), b.cuda())
        shared = moe.moe_grouped_gemm_act(*args, ws=ws)
        fresh = moe.moe_grouped_gemm_act(*args, ws=torch.zeros(256, dtype=torch.uint8,
                                                                device="cuda"))
        torch.cuda.synchronize()
        assert torch.equal(shared, fresh), f"case {i}: workspace reuse changed the result"
        assert int(ws[32:40].view(torch.int32).abs().sum()) == 0, "tile counters not reset"
        exact = O.grouped_gemm_act(np_(a), np_(w), np_(seg_end), F, spec["kind"],
                                   spec.get("swiglu_fusion", 2), spec.get("limit", 0.0),
                                   spec.get("alpha", 1.0), spec.get("beta", 0.0), np_(b),
                                   dtype=None)
        assert_rounded_once(np_(shared), exact, "bf16", f"pair kernel, shared workspace {i}")
        assert moe.moe_sync_status(ws) == moe.MOE_OK
