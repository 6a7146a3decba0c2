"""SwiGLU fusion 0 (gate from FC1, up from FC3, two weight tensors): the
split gate_up GEMM against the oracle and bit for bit against the stacked
layout holding the same two tensors (the accumulator tile and its k order are
the same), on the tcgen05 path, the SIMT path and fp32; the whole forward with
split weights bit for bit against the stacked forward and against the oracle."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

from gpu_cases import np_
from tolerances import assert_forward_close, assert_rounded_once

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


ACTS = {
    "swiglu0": dict(kind=1, swiglu_fusion=0, limit=7.0, alpha=1.702, beta=1.0),
    "swiglu0_noclamp": dict(kind=1, swiglu_fusion=0, limit=0.0, alpha=1.3, beta=0.5),
    "silu": dict(kind=0),
    "gelu_mul": dict(kind=3),
}


def _split_problem(counts, Hk, F, dtype, bias, seed):
    g = torch.Generator().manual_seed(seed)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    E, M = len(counts), int(sum(counts))
    a = torch.randn((M, Hk), generator=g).to(tdt)
    wg = (torch.randn((E, F, Hk), generator=g) / Hk ** 0.5).to(tdt)
    wu = (torch.randn((E, F, Hk), generator=g) / Hk ** 0.5).to(tdt)
    bg = (torch.randn((E, F), generator=g) * 0.02).to(tdt) if bias else None
    bu = (torch.randn((E, F), generator=g) * 0.02).to(tdt) if bias else None
    seg_end = torch.tensor(np.cumsum(counts), dtype=torch.int32)
    return a, wg, wu, bg, bu, seg_end


def _cu(t):
    return None if t is None else t.cuda()


@pytest.mark.parametrize("counts,Hk,F,act,bias,dtype,simt", [
    ([3, 0, 130, 1, 300], 256, 192, "swiglu0", True, "bf16", False),
    ([129, 127, 0, 256], 320, 160, "silu", False, "bf16", False),
    ([50, 0, 0, 77, 200], 200, 96, "gelu_mul", True, "bf16", False),   # ragged k-block
    ([200, 56, 100], 128, 136, "swiglu0_noclamp", True, "bf16", False),  # ragged column tile
    ([1], 64, 8, "swiglu0", False, "bf16", False),                       # one row
    ([129, 127, 0, 256], 320, 160, "swiglu0", True, "bf16", True),       # SIMT, bf16
    ([300, 5, 0, 211], 132, 36, "silu", True, "bf16", False),            # F % 8 != 0 -> SIMT
    ([40, 0, 25, 63], 100, 48, "swiglu0", True, "f32", False),           # fp32 (SIMT)
    ([129, 127, 0, 256], 320, 160, "swiglu0", True, "f16", False),       # float16 operands
])
def test_gemm_act_split(moe, counts, Hk, F, act, bias, dtype, simt):
    spec = ACTS[act]
    a, wg, wu, bg, bu, seg_end = _split_problem(counts, Hk, F, dtype, bias, seed=Hk * 7 + F)
    M = a.shape[0]
    p = moe.act_params(**spec)
    stacked = moe.act_params(**dict(spec, swiglu_fusion=2))
    out = torch.full((M + 5, F), float("nan"), dtype=a.dtype, device="cuda")
    ref = torch.full((M + 5, F), float("nan"), dtype=a.dtype, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    a_pad = torch.cat([a, torch.zeros((5, Hk), dtype=a.dtype)]).cuda()  # rows outside every segment
    old = moe.moe_set_gemm_simt(simt)
    try:
        moe.moe_grouped_gemm_act_split(a_pad, wg.cuda(), wu.cuda(), seg_end.cuda(), p, _cu(bg),
                                       _cu(bu), out=out, ws=ws)
        assert moe.moe_sync_status(ws) == moe.MOE_OK
        moe.moe_grouped_gemm_act(a_pad, torch.cat([wg, wu], 1).cuda(), seg_end.cuda(), F, stacked,
                                 None if bg is None else torch.cat([bg, bu], 1).cuda(), out=ref,
                                 ws=ws)
        assert moe.moe_sync_status(ws) == moe.MOE_OK
    finally:
        moe.moe_set_gemm_simt(old)
    got = np_(out)
    assert np.isnan(got[M:]).all(), "rows past the last segment were written"
    exact = O.grouped_gemm_act_split(np_(a), np_(wg), np_(wu), np_(seg_end), spec["kind"],
                                     spec.get("limit", 0.0), spec.get("alpha", 1.0),
                                     spec.get("beta", 0.0), None if bg is None else np_(bg),
                                     None if bu is None else np_(bu), dtype=None)
    assert_rounded_once(got[:M], exact, dtype, f"gemm_act_split {act}")
    np.testing.assert_array_equal(got[:M], np_(ref)[:M])


def test_split_rejects(moe):
    a, wg, wu, bg, bu, seg_end = _split_problem([4, 4], 64, 64, "bf16", True, seed=3)
    a, wg, wu, bg, bu, seg_end = (t.cuda() for t in (a, wg, wu, bg, bu, seg_end))
    for spec in (dict(kind=1, swiglu_fusion=1), dict(kind=1, swiglu_fusion=2), dict(kind=2),
                 dict(kind=4)):
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_grouped_gemm_act_split(a, wg, wu, seg_end, moe.act_params(**spec))
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoEError) as ei:  # one bias without the other
        moe.moe_grouped_gemm_act_split(a, wg, wu, seg_end, moe.act_params(kind=0), b_gate=bg)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("T,H,F,E,K,act,bias,dtype", [
    (300, 256, 192, 8, 2, "swiglu0", True, "bf16"),     # tcgen05, gathered rows
    (40, 128, 256, 16, 4, "silu", False, "bf16"),       # small T*K: still the staged path
    (200, 96, 72, 6, 2, "swiglu0_noclamp", True, "f32"),
    (300, 256, 192, 8, 2, "gelu_mul", True, "f16"),
])
def test_forward_split(moe, T, H, F, E, K, act, bias, dtype):
    spec = ACTS[act]
    g = torch.Generator().manual_seed(T + H + F)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    hidden = torch.randn((T, H), generator=g).to(tdt)
    logits = torch.randn((T, E), generator=g)
    wg = (torch.randn((E, F, H), generator=g) / H ** 0.5).to(tdt)
    wu = (torch.randn((E, F, H), generator=g) / H ** 0.5).to(tdt)
    wd = (torch.randn((E, H, F), generator=g) / F ** 0.5).to(tdt)
    bg = (torch.randn((E, F), generator=g) * 0.02).to(tdt) if bias else None
    bu = (torch.randn((E, F), generator=g) * 0.02).to(tdt) if bias else None
    bd = (torch.randn((E, H), generator=g) * 0.02).to(tdt) if bias else None
    rp = moe.route_params(top_k=K, scoring="softmax", renormalize=True)
    out = moe.moe_ffn_forward_split(hidden.cuda(), logits.cuda(), wg.cuda(), wu.cuda(), wd.cuda(),
                                    rp, moe.act_params(**spec), b_gate=_cu(bg), b_up=_cu(bu),
                                    b_down=_cu(bd))
    w1 = torch.cat([wg, wu], 1)
    b1 = None if bg is None else torch.cat([bg, bu], 1)
    ref = moe.moe_ffn_forward(hidden.cuda(), logits.cuda(), w1.cuda(), wd.cuda(), rp,
                              moe.act_params(**dict(spec, swiglu_fusion=2)), b_gate_up=_cu(b1),
                              b_down=_cu(bd))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(np_(out), np_(ref))
    r = O.ffn_forward(np_(hidden), np_(logits), np_(w1), np_(wd), b_gate_up=None if b1 is None
                      else np_(b1), b_down=None if bd is None else np_(bd), K=K, F=F,
                      scoring="softmax", renormalize=True, dtype=dtype, act=spec["kind"],
                      fusion=2, limit=spec.get("limit", 0.0), alpha=spec.get("alpha", 1.0),
                      beta=spec.get("beta", 0.0))
    assert_forward_close(np_(out), r, dtype, f"forward_split {act} {dtype}")


@pytest.mark.parametrize("name", ["qwen3_bf16", "gpt_oss_bf16"])
def test_forward_split_full_size(moe, name):
    """At the full workload sizes, in the forward's launch configuration: the
    forward with the two tensors is bit for bit the stacked forward."""
    from mixture_experts_ffn_gb300 import synth

    from gpu_cases import make

    cfg = synth.CONFIGS[name].replace(local_count=0)
    inp, _ = make(cfg)
    p, a = moe.config_params(cfg)
    F = cfg.F
    w1 = inp["w_gate_up"]
    b1 = inp["b_gate_up"]
    if a.swiglu_fusion == 1:  # interleaved rows: gate rows 2j, up rows 2j + 1
        wg, wu = w1[:, 0::2].contiguous(), w1[:, 1::2].contiguous()
        bg, bu = (None, None) if b1 is None else (b1[:, 0::2].contiguous(), b1[:, 1::2].contiguous())
    else:
        wg, wu = w1[:, :F].contiguous(), w1[:, F:].contiguous()
        bg, bu = (None, None) if b1 is None else (b1[:, :F].contiguous(), b1[:, F:].contiguous())
    a0 = moe.act_params(a.kind, 0 if a.kind == 1 else a.swiglu_fusion, a.limit, a.alpha, a.beta)
    out = moe.moe_ffn_forward_split(inp["hidden"], inp["logits"], wg, wu, inp["w_down"], p, a0,
                                    inp["correction_bias"], inp["expert_ids"], bg, bu,
                                    inp["b_down"])
    ref = moe.moe_ffn_forward(inp["hidden"], inp["logits"], w1, inp["w_down"], p, a,
                              inp["correction_bias"], inp["expert_ids"], b1, inp["b_down"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
