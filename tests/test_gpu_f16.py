"""float16 (the ORT MoE and MoERouter tensor type T = float16) against the
oracle: the grouped GEMMs on the tcgen05 path (kind::f16 with float16
operands) and the SIMT path, the combine, the standalone SwiGLU, the router
with float16 logits and its float16 router_probs (sentinel -1e4), the whole
forward, and an expert-parallel rank fed by float16 router_probs."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_gb300 import synth
from oracle import cases
from oracle import moe_oracle as O

from gpu_cases import np_
from tolerances import (assert_forward_close, assert_layer_close, assert_rounded_once, ulp_bf16,
                        ulp_f16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


def _guarded_logits(cfg, dtype):
    """[T, E] logits in ``dtype`` whose every row, as stored, keeps a routing
    margin >= cases.MIN_GAP (rows are redrawn until it does)."""
    tdt = synth.torch_dtype(dtype)
    z = synth.make_logits(cfg).to(tdt)
    cb = synth.make_correction_bias(cfg)
    bias = None if cb is None else cb.numpy()
    for attempt in range(1, 200):
        m = O.selection_margins(np_(z), cfg.K, cfg.scoring, cfg.G, cfg.TG, bias)
        bad = np.nonzero(m < cases.MIN_GAP)[0]
        if bad.size == 0:
            return z
        z[torch.from_numpy(bad)] = synth.make_logits(cfg, salt=attempt).to(tdt)[torch.from_numpy(bad)]
    raise RuntimeError("could not guard the logits")


@pytest.mark.parametrize("counts,Hk,F,spec,bias,simt", [
    ([3, 0, 130, 1, 300], 256, 192, dict(kind=0), True, False),
    ([129, 127, 0, 256], 320, 160, dict(kind=1, swiglu_fusion=1, limit=7.0, alpha=1.702,
                                        beta=1.0), True, False),
    ([200, 56, 100], 128, 384, dict(kind=2), True, False),                 # plain (identity)
    ([50, 0, 0, 77, 200], 200, 96, dict(kind=3), False, False),            # ragged k-block
    ([129, 127, 0, 256], 320, 160, dict(kind=0), True, True),              # SIMT
    ([300, 5, 0, 211], 132, 36, dict(kind=1, swiglu_fusion=2, limit=3.0), True, False),  # F%8
])
def test_gemm_act_f16(moe, counts, Hk, F, spec, bias, simt):
    g = torch.Generator().manual_seed(Hk + F)
    E, M = len(counts), int(sum(counts))
    N1 = 2 * F if spec["kind"] in (0, 1, 3) else F
    a = torch.randn((M, Hk), generator=g).half()
    w = (torch.randn((E, N1, Hk), generator=g) / Hk ** 0.5).half()
    b = (torch.randn((E, N1), generator=g) * 0.02).half() if bias else None
    seg_end = torch.tensor(np.cumsum(counts), dtype=torch.int32)
    out = torch.full((M, F), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    old = moe.moe_set_gemm_simt(simt)
    try:
        moe.moe_grouped_gemm_act(a.cuda(), w.cuda(), seg_end.cuda(), F, moe.act_params(**spec),
                                 None if b is None else b.cuda(), out=out, ws=ws)
        assert moe.moe_sync_status(ws) == moe.MOE_OK
    finally:
        moe.moe_set_gemm_simt(old)
    exact = O.grouped_gemm_act(np_(a), np_(w), np_(seg_end), F, spec["kind"],
                               spec.get("swiglu_fusion", 2), spec.get("limit", 0.0),
                               spec.get("alpha", 1.0), spec.get("beta", 0.0),
                               None if b is None else np_(b), dtype=None)
    assert_rounded_once(np_(out), exact, "f16", f"gemm_act f16 {spec}")


def test_gathered_and_down_f16(moe):
    """The gathered gate_up entry and the down GEMM in float16."""
    g = torch.Generator().manual_seed(5)
    T, K, H, F, E = 150, 2, 256, 128, 4
    hidden = torch.randn((T, H), generator=g).half()
    ids = torch.randint(0, E, (T, K), generator=g, dtype=torch.int32)
    r = O.permute(np_(ids), E)
    w1 = (torch.randn((E, 2 * F, H), generator=g) / H ** 0.5).half()
    w2 = (torch.randn((E, H, F), generator=g) / F ** 0.5).half()
    seg_end = torch.from_numpy(r["seg_end"].astype(np.int32))
    r2r = torch.from_numpy(r["row_to_route"].astype(np.int32))
    act = moe.moe_grouped_gemm_act_gathered(hidden.cuda(), r2r.cuda(), K, w1.cuda(),
                                            seg_end.cuda(), F, moe.act_params(kind=0))
    rows = np_(hidden)[r["row_to_route"] // K]
    exact = O.grouped_gemm_act(rows, np_(w1), r["seg_end"], F, 0, 2, dtype=None)
    assert_rounded_once(np_(act), exact, "f16", "gathered f16")
    y = moe.moe_grouped_gemm_down(act, w2.cuda(), seg_end.cuda())
    exact_y = O.grouped_gemm_down(np_(act), np_(w2), r["seg_end"], None, dtype=None)
    assert_rounded_once(np_(y), exact_y, "f16", "down f16")


def test_combine_and_swiglu_f16(moe):
    g = torch.Generator().manual_seed(9)
    T, K, H = 77, 4, 264  # H % 8 == 0: the 16-byte path; then H = 100: the scalar one
    for h in (H, 100):
        y = torch.randn((T * K, h), generator=g).half()
        w = torch.rand((T, K), generator=g)
        r2r = torch.randperm(T * K, generator=g).to(torch.int32)
        out = moe.moe_combine(y.cuda(), w.cuda(), r2r.cuda(), scale=1.5)
        exact = O.combine(np_(y), np_(w), np_(r2r), T, K, 1.5, dtype=None)
        assert_rounded_once(np_(out), exact, "f16", f"combine f16 H={h}")
    gate = torch.randn((33, 2 * 48), generator=g).half()
    out = moe.swiglu(gate.cuda(), None, swiglu_fusion=1, limit=7.0, alpha=1.702, beta=1.0)
    exact = O.swiglu_op(np_(gate), None, 48, 1, 7.0, 1.702, 1.0, dtype=None)
    assert_rounded_once(np_(out), exact, "f16", "swiglu f16")


@pytest.mark.parametrize("ldt", ["f16", "bf16"])
def test_route_16bit_logits_and_router_probs(moe, ldt):
    """Logits and router_probs in the MoERouter type T: ids equal to the
    oracle's on the same (widened) logits, router_probs equal to the oracle's
    rounded to T within one of T's ulps, and the sentinel -1e4 (f16) or
    -1e30 rounded to bf16 at every expert not chosen."""
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=1000)
    z = _guarded_logits(cfg, ldt)
    ls, lc = 32, 32
    p = moe.route_params(top_k=cfg.K, scoring="softmax", renormalize=True,
                         local_expert_start=ls, local_expert_count=lc, route_scale=1.0)
    tw, ti, probs, wsc = moe.moe_route(z.cuda(), p)
    assert probs.dtype == z.dtype
    r = O.route(np_(z), cfg.K, "softmax", True, local_start=ls, local_count=lc,
                probs_dtype=ldt)
    np.testing.assert_array_equal(np_(ti), r["topk_ids"])
    np.testing.assert_allclose(np_(tw), r["topk_weights"], rtol=1e-5)
    np.testing.assert_allclose(np_(wsc), r["weight_scale"], rtol=1e-5, atol=1e-7)
    got, want = np_(probs), r["router_probs"]
    sentinel = -1e4 if ldt == "f16" else float(O.round_to(np.array([-1e30]), "bf16")[0])
    np.testing.assert_array_equal(got == sentinel, want == sentinel)
    assert (want == sentinel).any() and (want != sentinel).any()
    live = want != sentinel
    ulp = ulp_f16(want[live]) if ldt == "f16" else ulp_bf16(want[live])
    assert (np.abs(got[live] - want[live]) <= ulp).all()


@pytest.mark.parametrize("T,ldt", [(512, "f32"), (300, "f16"), (4096, "f32")])
def test_forward_f16(moe, T, ldt):
    """The whole forward with float16 activations and weights (Qwen3-style
    shapes; the full 4096 tokens on a 256-token subset)."""
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=T, dtype="f16", local_start=0, local_count=0)
    z = _guarded_logits(cfg, ldt)
    inp = synth.make_inputs(cfg, "cuda", logits=z)
    p, a = moe.config_params(cfg)
    out = moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a)
    assert out.dtype == torch.float16
    tokens = None if T <= 512 else np.arange(0, T, T // 256)
    ref = O.ffn_forward(np_(inp["hidden"]), np_(z), np_(inp["w_gate_up"]), np_(inp["w_down"]),
                        K=cfg.K, F=cfg.F, scoring=cfg.scoring, renormalize=cfg.renormalize,
                        dtype="f16", tokens=tokens)
    got = np_(out) if tokens is None else np_(out)[tokens]
    assert_forward_close(got, ref, "f16", f"forward f16 T={T} logits {ldt}")


def test_local_forward_f16_router_probs(moe):
    """An expert-parallel rank fed by the oracle's float16 router_probs (with
    the -1e4 sentinel, tokens with no local expert included)."""
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=256, dtype="f16", E=32, K=4, F=256, H=512,
                                              local_start=0, local_count=0)
    z = _guarded_logits(cfg, "f32")
    inp = synth.make_inputs(cfg, "cuda", logits=z)
    lc, start = 8, 8
    r = O.route(np_(z), cfg.K, "softmax", True, local_start=start, local_count=lc,
                probs_dtype="f16")
    assert (r["weight_scale"] == 0).any()
    probs = torch.from_numpy(r["router_probs"]).half().cuda()
    wsc = torch.from_numpy(r["weight_scale"]).float().cuda()
    w1 = inp["w_gate_up"][start:start + lc].contiguous()
    w2 = inp["w_down"][start:start + lc].contiguous()
    out = moe.moe_ffn_forward_local(inp["hidden"], probs, wsc, w1, w2, cfg.K,
                                    moe.act_params(kind=0))
    ref = O.ffn_forward_local(np_(inp["hidden"]), r["router_probs"], np_(wsc), np_(w1), np_(w2),
                              cfg.K, cfg.F, dtype="f16", parts=True)
    assert_forward_close(np_(out), ref, "f16", "local forward f16", scale=r["weight_scale"])


def test_shared_expert_f16(moe):
    """The shared expert's dense gated MLP in float16 (one segment of T rows
    through the same tcgen05 GEMMs)."""
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=384, dtype="f16")
    hidden = torch.randn((cfg.T, cfg.H), generator=torch.Generator().manual_seed(4)).half()
    sw = synth.make_shared_expert(cfg, 512)
    out = moe.moe_shared_expert_mlp(hidden.cuda(), sw["shared_w_gate_up"].cuda(),
                                    sw["shared_w_down"].cuda())
    assert out.dtype == torch.float16
    exact = O.shared_expert_mlp(np_(hidden), np_(sw["shared_w_gate_up"]),
                                np_(sw["shared_w_down"]), dtype="f16", unrounded=True)
    assert_layer_close(np_(out), exact, "f16", "shared expert f16")
