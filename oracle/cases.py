"""Test cases built from the seeded generator plus the oracle's tie guard.

TEST INFRASTRUCTURE (see the package docstring for who may import it).

A routing decision computed in float32 on two machines can differ when two
selection scores are within a few ulp of each other.  ``guarded_logits``
redraws every token row whose decision margin (K-th vs (K+1)-th allowed
selection score, and TG-th vs (TG+1)-th group score) is below ``min_gap``
(1e-3), from independent seeded draws, so that the GPU and the oracle must
agree bit for bit on the routing.
"""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_ffn_gb300 import synth

from .moe_oracle import selection_margins

MIN_GAP = 1e-3


def guarded_logits(cfg: synth.MoEConfig, min_gap: float = MIN_GAP, max_attempts: int = 200):
    """[T, E] fp32 logits (CPU tensor) with every row's routing margin >= min_gap."""
    logits = synth.make_logits(cfg)
    if cfg.T == 0:
        return logits
    cb = synth.make_correction_bias(cfg)
    bias = None if cb is None else cb.numpy()
    for attempt in range(1, max_attempts + 1):
        m = selection_margins(logits.numpy(), cfg.K, cfg.scoring, cfg.G, cfg.TG, bias)
        bad = np.nonzero(m < min_gap)[0]
        if bad.size == 0:
            return logits
        fresh = synth.make_logits(cfg, salt=attempt)
        logits[torch.from_numpy(bad)] = fresh[torch.from_numpy(bad)]
    raise RuntimeError(f"could not guard {cfg.name}: {bad.size} rows left")


def oracle_kwargs(cfg: synth.MoEConfig) -> dict:
    """Keyword arguments of ``ffn_forward`` / ``route`` for a config."""
    return dict(K=cfg.K, scoring=cfg.scoring, renormalize=cfg.renormalize, G=cfg.G, TG=cfg.TG,
                rsf=cfg.rsf)


def to_np(t):
    """float64 / int numpy copy of a tensor (bf16 converts exactly)."""
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    a = t.numpy()
    return a.astype(np.float64) if a.dtype.kind == "f" else a
