"""The whole forward through moe_ffn_forward against the oracle, on every
workload recipe: reduced sizes (all tokens checked) and the full sizes the
benchmark runs (routing and permutation on all tokens, outputs on the fixed
256-token subset for the large recipes), plus the indexed decode path, the
dispatch rule, determinism and the device status word."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_gb300 import synth
from oracle import moe_oracle as O

from gpu_cases import act_kwargs, make, np_
from tolerances import assert_forward_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


def run_forward(moe, cfg, inp):
    p, a = moe.config_params(cfg)
    T = cfg.T
    tw = torch.empty((T, cfg.K), dtype=torch.float32, device="cuda")
    ti = torch.empty((T, cfg.K), dtype=torch.int32, device="cuda")
    probs = wsc = None
    if cfg.local_count:
        probs = torch.empty((T, cfg.local_count), dtype=torch.float32, device="cuda")
        wsc = torch.empty((T,), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.moe_workspace_size(T, cfg.H, cfg.F, cfg.E, cfg.K,
                                            {"bf16": moe.MOE_BF16, "f16": moe.MOE_F16,
                                             "f32": moe.MOE_F32}[cfg.dtype]),
                     dtype=torch.uint8, device="cuda")
    moe.moe_clear_status(ws)
    out = moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a,
                              inp["correction_bias"], inp["expert_ids"], inp["b_gate_up"],
                              inp["b_down"], topk_weights_out=tw, topk_ids_out=ti,
                              router_probs=probs, weight_scale=wsc, ws=ws)
    status = moe.moe_sync_status(ws)
    return out, tw, ti, probs, wsc, status


def oracle_forward(cfg, ref, tokens=None):
    return O.ffn_forward(ref["hidden"], ref["logits"], ref["w_gate_up"], ref["w_down"],
                         correction_bias=ref["correction_bias"], expert_ids=ref["expert_ids"],
                         b_gate_up=ref["b_gate_up"], b_down=ref["b_down"], K=cfg.K, F=cfg.F,
                         scoring=cfg.scoring, renormalize=cfg.renormalize, G=cfg.G, TG=cfg.TG,
                         rsf=cfg.rsf, dtype=cfg.dtype, local_start=cfg.local_start,
                         local_count=cfg.local_count, route_scale=cfg.route_scale, tokens=tokens,
                         **act_kwargs(cfg))


def check(moe, cfg, tokens=None, what=None):
    inp, ref = make(cfg)
    out, tw, ti, probs, wsc, status = run_forward(moe, cfg, inp)
    assert status == moe.MOE_OK
    # routing on all tokens
    r_all = O.route(ref["logits"], cfg.K, cfg.scoring, cfg.renormalize, cfg.G, cfg.TG, cfg.rsf,
                    ref["correction_bias"], ref["expert_ids"], cfg.local_start, cfg.local_count,
                    cfg.route_scale)
    np.testing.assert_array_equal(np_(ti), r_all["topk_ids"])
    np.testing.assert_allclose(np_(tw), r_all["topk_weights"], rtol=1e-5)
    if cfg.local_count:
        sent = r_all["router_probs"] == -1e30
        got = np_(probs)
        np.testing.assert_array_equal(got == np.float32(-1e30), sent)
        np.testing.assert_allclose(got[~sent], r_all["router_probs"][~sent], atol=1e-5)
        np.testing.assert_allclose(np_(wsc), r_all["weight_scale"], rtol=1e-5, atol=1e-7)
    # outputs on the token subset
    r = oracle_forward(cfg, ref, tokens)
    tok = r["tokens"]
    got = np_(out)[tok]
    what = what or cfg.name
    return assert_forward_close(got, r, cfg.dtype, what), out


SMALL = {
    "tiny_fp32": {},
    "qwen3_bf16": dict(T=300, H=256, F=192, E=32, K=8, local_start=8, local_count=8),
    "deepseek_v3_bf16": dict(T=300, H=320, F=128, E=64, K=8, G=8, TG=4),
    "gpt_oss_bf16": dict(T=200, H=192, F=160, E=16, K=4),
    "kimi_k2_decode_bf16": dict(T=16, H=256, F=256, E=96, K=8),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_ffn_small(moe, name):
    cfg = synth.CONFIGS[name].replace(**SMALL[name])
    check(moe, cfg, what=f"small {name}")


@pytest.mark.parametrize("name,over", [
    ("qwen3_bf16", dict(T=300, H=256, F=128, act=synth.ACT_GELU_AND_MUL,
                        scoring="sqrt_softplus")),                    # gathered gate_up
    ("gpt_oss_bf16", dict(T=200, H=256, F=128, act=synth.ACT_GELU, swiglu_fusion=2)),  # non-gated
    ("tiny_fp32", dict(act=synth.ACT_RELU)),                          # SIMT, fp32
    ("deepseek_v3_bf16", dict(T=256, H=256, F=128, act=synth.ACT_SILU,
                              scoring="sqrt_softplus")),              # bias + groups
])
def test_ffn_activation_and_scoring_variants(moe, name, over):
    """gelu_and_mul, the non-gated relu / gelu / silu and sqrt_softplus
    scoring through the whole forward against the oracle."""
    check(moe, synth.CONFIGS[name].replace(**over), what=f"variant {name} act {over.get('act')}")


def test_ffn_small_hash_routing(moe):
    cfg = synth.CONFIGS["kimi_k2_decode_bf16"].replace(hash_ids=True, T=16, H=256, F=256, E=96)
    check(moe, cfg, what="small kimi_k2_decode_bf16 hash")


@pytest.mark.parametrize("name,hash_ids", [
    ("tiny_fp32", False),
    ("qwen3_bf16", False),
    ("gpt_oss_bf16", False),
    ("kimi_k2_decode_bf16", False),
    ("kimi_k2_decode_bf16", True),
    ("deepseek_v3_bf16", False),
])
def test_ffn_full_size(moe, name, hash_ids):
    cfg = synth.CONFIGS[name].replace(hash_ids=hash_ids)
    tokens = None if cfg.T <= 4096 else synth.subset_tokens(cfg.T)
    if name == "gpt_oss_bf16":
        tokens = synth.subset_tokens(cfg.T)
    rep, _ = check(moe, cfg, tokens, what=f"full {name}{' hash' if hash_ids else ''}")
    print(name, rep)


@pytest.mark.parametrize("name", ["gpt_oss_bf16", "deepseek_v3_bf16", "kimi_k2_decode_bf16"])
def test_ffn_full_size_float16(moe, name):
    """The other recipes at their full sizes with float16 operands (the
    decode recipe then takes the staged path: the indexed kernel is bf16),
    on the fixed token subset."""
    cfg = synth.CONFIGS[name].replace(dtype="f16")
    tokens = None if cfg.T <= 256 else synth.subset_tokens(cfg.T)
    rep, _ = check(moe, cfg, tokens, what=f"full {name} f16")
    print(name, "f16", rep)


def test_indexed_path_matches_staged(moe):
    """The decode recipe satisfies the dispatch rule; the indexed kernels and the
    staged pipeline compute the same layer (both checked against the oracle)."""
    cfg = synth.CONFIGS["kimi_k2_decode_bf16"].replace(H=1024, F=512, E=64)
    inp, ref = make(cfg)
    p, a = moe.config_params(cfg)
    w, ids, _, _ = moe.moe_route(inp["logits"], p, inp["correction_bias"])
    y_idx = moe.moe_indexed_mlp(inp["hidden"], inp["w_gate_up"], inp["w_down"], w, ids)
    perm = moe.moe_permute(ids, cfg.E, inp["hidden"])
    act = moe.moe_grouped_gemm_act(perm["expert_input"], inp["w_gate_up"], perm["seg_end"], cfg.F, a)
    y = moe.moe_grouped_gemm_down(act, inp["w_down"], perm["seg_end"])
    y_st = moe.moe_combine(y, w, perm["route_to_row"])
    torch.cuda.synchronize()
    r = oracle_forward(cfg, ref)
    assert_forward_close(np_(y_idx), r, "bf16", "indexed vs oracle")
    assert_forward_close(np_(y_st), r, "bf16", "staged vs oracle")


def test_indexed_path_many_routes_per_expert(moe):
    """The indexed kernels take an expert's routes eight at a time: fixed ids
    that give experts 0..3 every token (27 routes each: three full passes and
    a tail of three) and spread the rest, checked against the oracle."""
    cfg = synth.CONFIGS["kimi_k2_decode_bf16"].replace(T=27, H=1024, F=512, E=16, K=6,
                                                       hash_ids=True)
    inp, ref = make(cfg)
    t = torch.arange(cfg.T, dtype=torch.int32).unsqueeze(1)
    tail = torch.stack([4 + (t[:, 0] % 6), 10 + (t[:, 0] % 6)], dim=1)
    ids = torch.cat([torch.arange(4, dtype=torch.int32).expand(cfg.T, 4), tail], dim=1)
    inp["expert_ids"] = ids.contiguous().cuda()
    ref["expert_ids"] = ids.numpy()
    p, a = moe.config_params(cfg)
    w, ids_out, _, _ = moe.moe_route(inp["logits"], p, inp["correction_bias"], inp["expert_ids"])
    y_idx = moe.moe_indexed_mlp(inp["hidden"], inp["w_gate_up"], inp["w_down"], w, ids_out)
    torch.cuda.synchronize()
    assert torch.equal(ids_out.cpu(), ids), "fixed ids not passed through"
    r = oracle_forward(cfg, ref)
    assert_forward_close(np_(y_idx), r, "bf16", "indexed, 27 routes per expert")


def test_forward_is_deterministic(moe):
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=512, H=512, F=256, E=64)
    inp, _ = make(cfg)
    o1 = run_forward(moe, cfg, inp)[0].clone()
    o2 = run_forward(moe, cfg, inp)[0]
    assert torch.equal(o1, o2)


def test_forward_bad_hash_ids_latch_device_error(moe):
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=64, H=128, F=64, E=16, K=2, local_count=0)
    inp, _ = make(cfg)
    ids = torch.randint(0, 16, (64, 2), dtype=torch.int32, device="cuda")
    ids[5, 1] = 99
    inp["expert_ids"] = ids
    *_, status = run_forward(moe, cfg, inp)
    assert status == moe.MOE_ERR_DEVICE


def test_forward_rejects_overlap_without_writing(moe):
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=64, H=128, F=64, E=16, K=2, local_count=0)
    inp, _ = make(cfg)
    p, a = moe.config_params(cfg)
    before = inp["hidden"].clone()
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a,
                            out=inp["hidden"])
    assert ei.value.status == moe.MOE_ERR_OVERLAP
    assert torch.equal(before, inp["hidden"])


def test_empty_batch(moe):
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=0, H=128, F=64, E=16, K=2, local_count=0)
    inp, _ = make(cfg, guard=False)
    p, a = moe.config_params(cfg)
    out = moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a)
    assert out.shape == (0, 128)


def test_concurrent_forwards_on_two_streams(moe):
    """Two forwards enqueued alternately on two streams (each with its own
    workspace) run concurrently on the GPU: both finish with status OK and
    give, bit for bit, the output of a forward run alone."""
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=512, H=256, F=128, E=32, K=8, local_count=0)
    inp, _ = make(cfg)
    p, a = moe.config_params(cfg)
    dt = moe.MOE_BF16
    ref = moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [torch.zeros(moe.moe_workspace_size(cfg.T, cfg.H, cfg.F, cfg.E, cfg.K, dt),
                       dtype=torch.uint8, device="cuda") for _ in streams]
    outs = [torch.empty_like(ref) for _ in streams]
    for _ in range(40):
        for s, ws, o in zip(streams, wss, outs):
            with torch.cuda.stream(s):
                moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"],
                                    inp["w_down"], p, a, out=o, ws=ws)
    torch.cuda.synchronize()
    for ws, o in zip(wss, outs):
        assert moe.moe_sync_status(ws) == moe.MOE_OK
        assert torch.equal(o, ref)


@pytest.mark.parametrize("name,over", [
    ("qwen3_bf16", dict(T=300, H=256, F=128, local_count=0)),        # gathered gate_up
    ("gpt_oss_bf16", dict(T=200, H=256, F=128)),                     # gathered, biases, SwiGLU
    ("tiny_fp32", dict()),                                           # staged, SIMT GEMMs
    ("kimi_k2_decode_bf16", dict(T=8, H=256, F=256)),                # indexed decode path
])
@pytest.mark.parametrize("pinned", [True, False])
def test_forward_host_matches_device(moe, name, over, pinned):
    """moe_ffn_forward_host (host activations and result; the activation copy
    on a side stream, the result written in place when it is page-locked)
    equals moe_ffn_forward on device copies of the same inputs bit for bit,
    with a page-locked or a pageable result buffer."""
    cfg = synth.CONFIGS[name].replace(**over)
    inp, _ = make(cfg)
    p, a = moe.config_params(cfg)
    ref = moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a,
                              inp["correction_bias"], inp["expert_ids"], inp["b_gate_up"],
                              inp["b_down"])
    h_host = inp["hidden"].cpu()
    l_host = inp["logits"].cpu()
    o_host = torch.full(tuple(ref.shape), float("nan"), dtype=ref.dtype)
    if pinned:
        h_host, l_host, o_host = h_host.pin_memory(), l_host.pin_memory(), o_host.pin_memory()
    dt = moe.MOE_BF16 if cfg.dtype == "bf16" else moe.MOE_F32
    ws = moe._ws(moe.moe_workspace_size_host(cfg.T, cfg.H, cfg.F, cfg.E, cfg.K, dt), "cuda")
    for _ in range(2):  # the second call reuses the side stream and the workspace
        o_host.fill_(float("nan"))
        moe.moe_ffn_forward_host(h_host, l_host, inp["w_gate_up"], inp["w_down"], p, a, o_host, ws,
                                 inp["correction_bias"], inp["expert_ids"], inp["b_gate_up"],
                                 inp["b_down"])
        assert moe.moe_sync_status(ws) == moe.MOE_OK
        assert torch.equal(o_host, ref.cpu())
