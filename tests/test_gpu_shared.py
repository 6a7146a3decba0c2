"""The shared expert (TileOPs "MoE Operators", SharedExpertMLPFwdOp) and the
shared + routed forward (FusedMoESharedExpertFwdOp, tp_size 1) against the
oracle: reduced sizes with every token checked, ragged token counts, the SIMT
fallbacks, a DeepSeek-V3-sized shared expert on sampled tokens, and the
two outputs of the fused op apart."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_gb300 import synth
from oracle import moe_oracle as O

from gpu_cases import act_kwargs, make, np_
from tolerances import assert_forward_close, assert_layer_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


@pytest.mark.parametrize("name,T,H,S", [
    ("qwen3_bf16", 300, 256, 384),     # tensor cores; 3 row tiles, ragged tail
    ("qwen3_bf16", 1, 64, 64),         # one token
    ("qwen3_bf16", 1000, 512, 256),
    ("qwen3_bf16", 40, 96, 36),        # S % 8 != 0: the exact-fp32 SIMT GEMM
    ("tiny_fp32", 50, 40, 24),         # fp32 (SIMT)
])
def test_shared_expert_mlp(moe, name, T, H, S):
    cfg = synth.CONFIGS[name].replace(T=T, H=H)
    inp = synth.make_inputs(cfg, "cuda")
    sw = synth.make_shared_expert(cfg, S, "cuda")
    out = moe.moe_shared_expert_mlp(inp["hidden"], sw["shared_w_gate_up"], sw["shared_w_down"])
    mdt = moe.MOE_BF16 if cfg.dtype == "bf16" else moe.MOE_F32
    ws = moe._ws(moe.moe_shared_expert_workspace_size(T, H, S, mdt), "cuda")
    out2 = moe.moe_shared_expert_mlp(inp["hidden"], sw["shared_w_gate_up"], sw["shared_w_down"],
                                     ws=ws)
    assert moe.moe_sync_status(ws) == moe.MOE_OK
    assert torch.equal(out, out2), "not deterministic"
    want = O.shared_expert_mlp(np_(inp["hidden"]), np_(sw["shared_w_gate_up"]),
                               np_(sw["shared_w_down"]), dtype=cfg.dtype, unrounded=True)
    assert_layer_close(np_(out), want, cfg.dtype, f"shared expert {name} T={T} S={S}")


def test_shared_expert_deepseek_size_sampled(moe):
    """DeepSeek-V3-sized shared expert (T 8192, H 7168, S 2048) on the tensor
    cores; the oracle checks 64 tokens (each output row depends on its own
    token only)."""
    cfg = synth.CONFIGS["deepseek_v3_bf16"]
    hidden = synth.make_inputs(cfg.replace(E=1, F=8), "cuda")["hidden"]
    sw = synth.make_shared_expert(cfg, 2048, "cuda")
    out = moe.moe_shared_expert_mlp(hidden, sw["shared_w_gate_up"], sw["shared_w_down"])
    torch.cuda.synchronize()
    rows = synth.subset_tokens(cfg.T, 64)
    want = O.shared_expert_mlp(np_(hidden[rows]), np_(sw["shared_w_gate_up"]),
                               np_(sw["shared_w_down"]), dtype="bf16", unrounded=True)
    assert_layer_close(np_(out[rows]), want, "bf16", "shared expert DeepSeek-V3 size")


@pytest.mark.parametrize("name", ["qwen3_bf16", "deepseek_v3_bf16"])
def test_forward_shared(moe, name):
    """The fused op's routed output equals moe_ffn_forward and its shared
    output moe_shared_expert_mlp, bit for bit, and both match the oracle;
    without shared weights only the routed output is produced."""
    cfg = synth.CONFIGS[name].replace(T=257, H=256, F=128, local_count=0)
    inp, ref = make(cfg)
    S = 192
    sw = synth.make_shared_expert(cfg, S, "cuda")
    p, a = moe.config_params(cfg)
    shared, routed = moe.moe_ffn_forward_shared(inp["hidden"], inp["logits"], inp["w_gate_up"],
                                                inp["w_down"], p, a, inp["correction_bias"],
                                                sw["shared_w_gate_up"], sw["shared_w_down"])
    routed_ref = moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"],
                                     inp["w_down"], p, a, inp["correction_bias"])
    shared_ref = moe.moe_shared_expert_mlp(inp["hidden"], sw["shared_w_gate_up"],
                                           sw["shared_w_down"])
    torch.cuda.synchronize()
    assert torch.equal(routed, routed_ref)
    assert torch.equal(shared, shared_ref)
    o = O.ffn_forward_shared(ref["hidden"], ref["logits"], ref["w_gate_up"], ref["w_down"],
                             np_(sw["shared_w_gate_up"]), np_(sw["shared_w_down"]),
                             dtype=cfg.dtype, K=cfg.K, F=cfg.F, scoring=cfg.scoring,
                             renormalize=cfg.renormalize, G=cfg.G, TG=cfg.TG, rsf=cfg.rsf,
                             correction_bias=ref["correction_bias"], **act_kwargs(cfg))
    assert_forward_close(np_(routed), o, cfg.dtype, f"forward_shared {name} routed")
    assert_layer_close(np_(shared), o["shared_unrounded"], cfg.dtype,
                       f"forward_shared {name} shared")
    none, routed2 = moe.moe_ffn_forward_shared(inp["hidden"], inp["logits"], inp["w_gate_up"],
                                               inp["w_down"], p, a, inp["correction_bias"])
    torch.cuda.synchronize()
    assert none is None and torch.equal(routed2, routed_ref)


def test_shared_rejects_half_the_weights(moe):
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=8, H=64, F=32, local_count=0)
    inp, _ = make(cfg)
    sw = synth.make_shared_expert(cfg, 32, "cuda")
    p, a = moe.config_params(cfg)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_ffn_forward_shared(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"],
                                   p, a, None, sw["shared_w_gate_up"], None,
                                   shared_out=torch.empty_like(inp["hidden"]))
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
