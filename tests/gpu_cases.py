"""GPU-side inputs plus the oracle's numpy view of the same bytes."""
import numpy as np
import torch

from mixture_experts_ffn_gb300 import synth
from oracle import cases

BIG_WEIGHT_BYTES = 1 << 28  # draw weight stacks on the GPU above this size


class LazyExperts:
    """numpy view of one expert of a device weight stack, fetched on demand."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return self.t[int(e)].float().cpu().numpy()


def make(cfg, guard=True):
    """Inputs of ``cfg`` on cuda:0 and the oracle's view of them."""
    logits = cases.guarded_logits(cfg) if guard else None
    wbytes = cfg.E * (cfg.n_gate_up + cfg.F) * cfg.H * (4 if cfg.dtype == "f32" else 2)
    wdev = "cuda" if wbytes > BIG_WEIGHT_BYTES else "cpu"
    inp = synth.make_inputs(cfg, "cuda", weight_device=wdev, logits=logits)
    ref = {k: cases.to_np(v) for k, v in inp.items() if k not in ("w_gate_up", "w_down")}
    if wdev == "cpu":
        ref["w_gate_up"] = cases.to_np(inp["w_gate_up"])
        ref["w_down"] = cases.to_np(inp["w_down"])
    else:
        ref["w_gate_up"] = LazyExperts(inp["w_gate_up"])
        ref["w_down"] = LazyExperts(inp["w_down"])
    return inp, ref


def act_kwargs(cfg):
    return dict(act=cfg.act, fusion=cfg.swiglu_fusion, limit=cfg.limit, alpha=cfg.alpha,
                beta=cfg.beta)


def np_(t):
    return cases.to_np(t)
