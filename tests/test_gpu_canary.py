"""Canary-padded outputs: every output of a call, and its workspace, is a
slice in the middle of a larger buffer filled with a sentinel, and after the
call the regions before and after each slice must still hold the sentinel
(no kernel writes outside what it was given).  Covers the whole forward on
each workload recipe at reduced size (staged, gathered, indexed and fp32
paths, the MoERouter slice outputs), and the stage calls one by one."""
import math

import pytest
import torch

from mixture_experts_ffn_gb300 import synth

from gpu_cases import make

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements of sentinel on each side (a multiple of 256 bytes for every dtype)


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


class Guarded:
    """A tensor of `shape` inside a sentinel-filled buffer."""

    def __init__(self, shape, dtype):
        self.n = math.prod(shape)
        self.fill = -7 if dtype in (torch.int32, torch.uint8) else float("nan")
        self.buf = torch.full((GUARD + self.n + GUARD,), self.fill, dtype=dtype, device="cuda")
        self.t = self.buf[GUARD:GUARD + self.n].view(shape)

    def intact(self):
        for part in (self.buf[:GUARD], self.buf[GUARD + self.n:]):
            if isinstance(self.fill, float):
                if not torch.isnan(part).all():
                    return False
            elif not (part == self.fill).all():
                return False
        return True


def guarded_ws(nbytes):
    # 256-byte aligned (torch allocations are 512-byte aligned and GUARD bytes
    # of uint8 sentinel come first); the status area starts cleared
    g = Guarded((max(nbytes, 256),), torch.uint8)
    g.t[:256].zero_()
    return g


def _dt(moe, cfg):
    return {"bf16": moe.MOE_BF16, "f16": moe.MOE_F16, "f32": moe.MOE_F32}[cfg.dtype]


@pytest.mark.parametrize("name,over", [
    ("qwen3_bf16", dict(T=200, H=256, F=192, E=32, local_start=8, local_count=16)),  # MoERouter
    ("deepseek_v3_bf16", dict(T=96, H=256, F=128, E=32)),         # grouped top-k
    ("deepseek_v3_bf16", dict(T=512, H=2048, F=256, E=8, G=1, TG=1)),  # SM-pair gate_up
    ("gpt_oss_bf16", dict(T=64, H=192, F=160, E=16)),             # biases, interleaved SwiGLU
    ("kimi_k2_decode_bf16", dict(T=8, H=1024, F=512, E=64)),      # indexed path
    ("tiny_fp32", dict()),                                        # fp32 staged path
])
def test_forward_writes_only_its_outputs(moe, name, over):
    cfg = synth.CONFIGS[name].replace(**over)
    inp, _ = make(cfg)
    p, a = moe.config_params(cfg)
    T, H, K = cfg.T, cfg.H, cfg.K
    tdt = inp["hidden"].dtype
    out = Guarded((T, H), tdt)
    tw = Guarded((T, K), torch.float32)
    ti = Guarded((T, K), torch.int32)
    probs = Guarded((T, cfg.local_count), torch.float32) if cfg.local_count else None
    wsc = Guarded((T,), torch.float32) if cfg.local_count else None
    ws = guarded_ws(moe.moe_workspace_size(T, H, cfg.F, cfg.E, K, _dt(moe, cfg)))
    moe.moe_ffn_forward(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p, a,
                        inp["correction_bias"], inp["expert_ids"], inp["b_gate_up"],
                        inp["b_down"], out=out.t, topk_weights_out=tw.t, topk_ids_out=ti.t,
                        router_probs=None if probs is None else probs.t,
                        weight_scale=None if wsc is None else wsc.t, ws=ws.t)
    assert moe.moe_sync_status(ws.t) == moe.MOE_OK
    torch.cuda.synchronize()
    for what, g in (("out", out), ("topk_weights", tw), ("topk_ids", ti), ("router_probs", probs),
                    ("weight_scale", wsc), ("workspace", ws)):
        if g is not None:
            assert g.intact(), f"{name}: wrote outside {what}"
    assert not torch.isnan(out.t.float()).any(), f"{name}: out not fully written"


def test_stage_calls_write_only_their_outputs(moe):
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=300, H=512, F=256, E=16, local_start=4,
                                              local_count=8)
    inp, _ = make(cfg)
    p, a = moe.config_params(cfg)
    T, H, F, E, K = cfg.T, cfg.H, cfg.F, cfg.E, cfg.K
    M = T * K
    tdt = inp["hidden"].dtype

    # router with its MoERouter slice
    tw, ti = Guarded((T, K), torch.float32), Guarded((T, K), torch.int32)
    probs, wsc = Guarded((T, cfg.local_count), torch.float32), Guarded((T,), torch.float32)
    moe.moe_route(inp["logits"], p, inp["correction_bias"], None, topk_weights=tw.t,
                  topk_ids=ti.t, router_probs=probs.t, weight_scale=wsc.t)
    torch.cuda.synchronize()
    assert all(g.intact() for g in (tw, ti, probs, wsc)), "moe_route wrote outside its outputs"

    # index maps, gathered gate_up, down, combine, standalone SwiGLU
    perm = moe.moe_permute(ti.t, E, inp["hidden"])
    act = Guarded((M, F), tdt)
    ws = guarded_ws(256)
    moe.moe_grouped_gemm_act_gathered(inp["hidden"], perm["row_to_route"], K, inp["w_gate_up"],
                                      perm["seg_end"], F, a, inp["b_gate_up"], out=act.t, ws=ws.t)
    y = Guarded((M, H), tdt)
    moe.moe_grouped_gemm_down(act.t, inp["w_down"], perm["seg_end"], inp["b_down"], out=y.t,
                              ws=ws.t)
    out = Guarded((T, H), tdt)
    moe.moe_combine(y.t, tw.t, perm["route_to_row"], out=out.t)
    gate = torch.randn((M, 2 * F), device="cuda").to(tdt)
    sg = Guarded((M, F), tdt)
    moe.swiglu(gate, None, 1, 7.0, 1.702, 1.0, out=sg.t)
    assert moe.moe_sync_status(ws.t) == moe.MOE_OK
    torch.cuda.synchronize()
    for what, g in (("gate_up", act), ("down", y), ("combine", out), ("swiglu", sg),
                    ("workspace", ws)):
        assert g.intact(), f"wrote outside {what}"
        if what != "workspace":
            assert not torch.isnan(g.t.float()).any(), f"{what} not fully written"


def test_shared_and_local_forwards_write_only_their_outputs(moe):
    """The shared expert alone, the shared + routed forward (two outputs) and
    an expert-parallel rank's forward from its MoERouter outputs."""
    cfg = synth.CONFIGS["deepseek_v3_bf16"].replace(T=100, H=256, F=128, E=32, local_start=8,
                                                    local_count=8)
    inp, _ = make(cfg)
    p, a = moe.config_params(cfg)
    T, H, F, E, K, S = cfg.T, cfg.H, cfg.F, cfg.E, cfg.K, 192
    tdt = inp["hidden"].dtype
    g = torch.Generator(device="cuda").manual_seed(5)
    sw1 = (torch.randn((2 * S, H), device="cuda", generator=g) / H ** 0.5).to(tdt)
    sw2 = (torch.randn((H, S), device="cuda", generator=g) / S ** 0.5).to(tdt)
    lib = moe.load_library()

    so = Guarded((T, H), tdt)
    ws1 = guarded_ws(lib.moe_shared_expert_workspace_size(T, H, S, moe.MOE_BF16))
    moe.moe_shared_expert_mlp(inp["hidden"], sw1, sw2, out=so.t, ws=ws1.t)

    ro, so2 = Guarded((T, H), tdt), Guarded((T, H), tdt)
    ws2 = guarded_ws(lib.moe_workspace_size_shared(T, H, F, S, E, K, moe.MOE_BF16))
    p0, _ = moe.config_params(cfg.replace(local_count=0))  # (no MoERouter outputs here)
    moe.moe_ffn_forward_shared(inp["hidden"], inp["logits"], inp["w_gate_up"], inp["w_down"], p0,
                               a, inp["correction_bias"], sw1, sw2, routed_out=ro.t,
                               shared_out=so2.t, ws=ws2.t)

    _, _, probs, wsc = moe.moe_route(inp["logits"], p, inp["correction_bias"])
    ls, lc = cfg.local_start, cfg.local_count
    lo = Guarded((T, H), tdt)
    ws3 = guarded_ws(lib.moe_workspace_size(T, H, F, lc, min(K, lc), moe.MOE_BF16))
    moe.moe_ffn_forward_local(inp["hidden"], probs, wsc, inp["w_gate_up"][ls:ls + lc].contiguous(),
                              inp["w_down"][ls:ls + lc].contiguous(), K, a, out=lo.t, ws=ws3.t)
    for ws in (ws1, ws2, ws3):
        assert moe.moe_sync_status(ws.t) == moe.MOE_OK
    torch.cuda.synchronize()
    for what, gd in (("shared_mlp", so), ("routed", ro), ("shared", so2), ("local", lo),
                     ("shared workspace", ws1), ("shared+routed workspace", ws2),
                     ("local workspace", ws3)):
        assert gd.intact(), f"wrote outside {what}"
        if "workspace" not in what:
            assert not torch.isnan(gd.t.float()).any(), f"{what} not fully written"
