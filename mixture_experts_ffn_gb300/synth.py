"""Seeded synthetic inputs for the routed MoE FFN forward.

This module only draws random numbers: it holds none of the method's
arithmetic (no scoring, no selection, no GEMM).  Both the CUDA path (bench,
tests) and the CPU oracle (tests) take their inputs from here, so the two sides
see the same bytes.

Recipes follow the model-shaped workloads named for this library:

* ``tiny_fp32``     T=64   H=128  F=64   E=8   K=2  fp32, softmax, silu_and_mul
* ``qwen3_bf16``    T=4096 H=2048 F=768  E=128 K=8  softmax, silu_and_mul,
                    MoERouter slice [32, 64)
* ``deepseek_v3_bf16`` T=8192 H=7168 F=2048 E=256 K=8 sigmoid + correction
                    bias, 8 groups / 4 kept, rsf 2.5
* ``gpt_oss_bf16``  T=2048 H=2880 F=2880 E=128 K=4 softmax, clamped SwiGLU
                    interleaved (limit 7, alpha 1.702, beta 1), both biases
* ``kimi_k2_decode_bf16`` T=16 H=7168 F=2048 E=384 K=8 sigmoid + correction
                    bias, rsf 2.827, optional fixed expert ids (hash routing)

Distributions: hidden ~ N(0,1); logits ~ N(0, sigma) fp32; weights ~
N(0, 1/sqrt(fan_in)) with fan_in = H for w_gate_up and F for w_down; biases ~
N(0, 0.02); correction bias ~ N(0, 0.1).  Every "N(0, s)" is read as standard
deviation s.  Each tensor has its own ``torch.Generator`` seeded with
``1000 * config_index + tensor_id`` (the tiny config has index 0, so its base
seed is 0); row redraws add ``1_000_000 * attempt``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

# tensor ids used in the per-tensor seed
TID_HIDDEN, TID_LOGITS, TID_W1, TID_W2, TID_CBIAS, TID_B1, TID_B2, TID_IDS = range(8)
TID_SW1, TID_SW2 = 8, 9  # shared-expert weights

# activation kinds (mirror the values of the C header's moe_act_kind)
ACT_SILU_AND_MUL = 0
ACT_SWIGLU = 1
ACT_IDENTITY = 2
ACT_GELU_AND_MUL = 3
ACT_RELU, ACT_GELU, ACT_SILU = 4, 5, 6
GATED_ACTS = (ACT_SILU_AND_MUL, ACT_SWIGLU, ACT_GELU_AND_MUL)


@dataclasses.dataclass
class MoEConfig:
    name: str
    index: int  # seed base = 1000 * index
    T: int
    H: int
    F: int
    E: int
    K: int
    dtype: str = "bf16"  # "bf16", "f16" or "f32"
    scoring: str = "softmax"  # "softmax" or "sigmoid"
    renormalize: bool = True
    G: int = 1  # num_expert_group
    TG: int = 1  # topk_group
    rsf: float = 1.0  # routed_scaling_factor
    act: int = ACT_SILU_AND_MUL
    swiglu_fusion: int = 2  # 1 interleaved, 2 concatenated / stacked
    limit: float = 0.0
    alpha: float = 1.0
    beta: float = 0.0
    logit_std: float = 1.0
    cbias_std: Optional[float] = None  # correction bias std, None = no bias
    bias_std: Optional[float] = None  # b_gate_up / b_down std, None = none
    hash_ids: bool = False  # pass fixed expert_ids
    local_start: int = 0
    local_count: int = 0  # 0 = no MoERouter outputs
    route_scale: float = 1.0

    @property
    def M(self) -> int:
        return self.T * self.K

    @property
    def n_gate_up(self) -> int:
        """Rows of w_gate_up per expert: 2F for gated activations, F otherwise."""
        return 2 * self.F if self.act in GATED_ACTS else self.F

    def replace(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny_fp32": MoEConfig("tiny_fp32", 0, T=64, H=128, F=64, E=8, K=2, dtype="f32",
                           scoring="softmax", renormalize=True, logit_std=1.0),
    "qwen3_bf16": MoEConfig("qwen3_bf16", 1, T=4096, H=2048, F=768, E=128, K=8,
                            scoring="softmax", renormalize=True, logit_std=2.0,
                            local_start=32, local_count=32, route_scale=1.0),
    "deepseek_v3_bf16": MoEConfig("deepseek_v3_bf16", 2, T=8192, H=7168, F=2048, E=256, K=8,
                                  scoring="sigmoid", renormalize=True, G=8, TG=4, rsf=2.5,
                                  logit_std=1.0, cbias_std=0.1),
    "gpt_oss_bf16": MoEConfig("gpt_oss_bf16", 3, T=2048, H=2880, F=2880, E=128, K=4,
                              scoring="softmax", renormalize=True, act=ACT_SWIGLU,
                              swiglu_fusion=1, limit=7.0, alpha=1.702, beta=1.0,
                              logit_std=1.0, bias_std=0.02),
    "kimi_k2_decode_bf16": MoEConfig("kimi_k2_decode_bf16", 4, T=16, H=7168, F=2048, E=384,
                                     K=8, scoring="sigmoid", renormalize=True, G=1, rsf=2.827,
                                     logit_std=1.0, cbias_std=0.1),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[name]


def _gen(cfg: MoEConfig, tid: int, device, salt: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(1000 * cfg.index + tid + 1_000_000 * salt)
    return g


def _normal(shape, std: float, gen: torch.Generator, device, out_dtype) -> torch.Tensor:
    """N(0, std) drawn in fp32, scaled, then cast once to ``out_dtype``."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(out_dtype)


def _normal_rows(n_outer: int, inner_shape, std: float, gen, device, out_dtype) -> torch.Tensor:
    """Like ``_normal`` for shape [n_outer, *inner_shape], drawn one outer slice at a
    time so that large weight stacks never hold a full fp32 copy."""
    out = torch.empty((n_outer, *inner_shape), device=device, dtype=out_dtype)
    for i in range(n_outer):
        x = torch.randn(inner_shape, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out[i].copy_(x)
    return out


def make_logits(cfg: MoEConfig, salt: int = 0) -> torch.Tensor:
    """[T, E] fp32 router logits drawn on the CPU; ``salt`` > 0 gives an
    independent redraw (used to replace rows)."""
    return _normal((cfg.T, cfg.E), cfg.logit_std, _gen(cfg, TID_LOGITS, "cpu", salt), "cpu",
                   torch.float32)


def make_expert_ids(cfg: MoEConfig) -> torch.Tensor:
    """[T, K] int32 fixed expert ids: K distinct uniform ids per token."""
    g = _gen(cfg, TID_IDS, "cpu")
    rows = [torch.randperm(cfg.E, generator=g)[: cfg.K] for _ in range(cfg.T)]
    ids = torch.stack(rows).to(torch.int32) if rows else torch.empty((0, cfg.K), dtype=torch.int32)
    return ids


def make_correction_bias(cfg: MoEConfig):
    """[E] fp32 selection-only correction bias drawn on the CPU, or None."""
    if cfg.cbias_std is None:
        return None
    return _normal((cfg.E,), cfg.cbias_std, _gen(cfg, TID_CBIAS, "cpu"), "cpu", torch.float32)


def make_inputs(cfg: MoEConfig, device="cpu", weight_device=None, logits=None) -> dict:
    """All inputs of one forward call, placed on ``device``.

    Activations, logits and the small per-expert vectors are always drawn with
    CPU generators, so their bytes do not depend on ``device``.  The two weight
    stacks are drawn on ``weight_device`` (default: ``device``); drawing them on
    the GPU is much faster for the large configs, and gives different (equally
    seeded) bytes than a CPU draw.  ``logits`` overrides the drawn logits (the
    tests pass rows redrawn away from routing ties)."""
    dt = torch_dtype(cfg.dtype)
    wdev = device if weight_device is None else weight_device
    lg = make_logits(cfg) if logits is None else logits
    inp = {
        "hidden": _normal((cfg.T, cfg.H), 1.0, _gen(cfg, TID_HIDDEN, "cpu"), "cpu", dt),
        "logits": lg,
        "correction_bias": make_correction_bias(cfg),
        "expert_ids": None,
        "b_gate_up": None,
        "b_down": None,
    }
    n1 = cfg.n_gate_up
    if cfg.hash_ids:
        inp["expert_ids"] = make_expert_ids(cfg)
    if cfg.bias_std is not None:
        inp["b_gate_up"] = _normal((cfg.E, n1), cfg.bias_std, _gen(cfg, TID_B1, "cpu"), "cpu", dt)
        inp["b_down"] = _normal((cfg.E, cfg.H), cfg.bias_std, _gen(cfg, TID_B2, "cpu"), "cpu", dt)
    inp = {k: (None if v is None else v.to(device)) for k, v in inp.items()}
    inp["w_gate_up"] = _normal_rows(cfg.E, (n1, cfg.H), 1.0 / math.sqrt(cfg.H),
                                    _gen(cfg, TID_W1, wdev), wdev, dt).to(device)
    inp["w_down"] = _normal_rows(cfg.E, (cfg.H, cfg.F), 1.0 / math.sqrt(cfg.F),
                                 _gen(cfg, TID_W2, wdev), wdev, dt).to(device)
    return inp


def make_shared_expert(cfg: MoEConfig, S: int, device="cpu") -> dict:
    """Weights of a shared expert with intermediate size S for ``cfg``'s
    hidden size: w_gate_up [2S, H] (std 1/sqrt(H)) and w_down [H, S]
    (std 1/sqrt(S)), drawn on ``device`` in the operand dtype."""
    dt = torch_dtype(cfg.dtype)
    return {
        "shared_w_gate_up": _normal((2 * S, cfg.H), 1.0 / math.sqrt(cfg.H),
                                    _gen(cfg, TID_SW1, device), device, dt),
        "shared_w_down": _normal((cfg.H, S), 1.0 / math.sqrt(S), _gen(cfg, TID_SW2, device),
                                 device, dt),
    }


def _quantize_blocks(x: torch.Tensor, rows_per_block: int):
    """Block-scaled e4m3 codes of x [.., R, K] with one fp32 scale per
    rows_per_block rows x 128 columns: scale = amax / 448 (the largest finite
    e4m3 value), codes = x / scale rounded to float8_e4m3fn by torch."""
    *lead, R, K = x.shape
    xb = x.reshape(*lead, R // rows_per_block, rows_per_block, K // 128, 128)
    amax = xb.abs().amax(dim=(-3, -1)).clamp_min(1e-12)          # [.., R/rb, K/128]
    scale = (amax / 448.0).to(torch.float32)
    q = (xb / scale[..., :, None, :, None]).reshape(*lead, R, K).to(torch.float8_e4m3fn)
    return q, scale


def make_fp8_masked(E: int, max_m: int, N: int, K: int, seed: int, device="cpu",
                    counts=None) -> dict:
    """Inputs of the block-scaled FP8 masked grouped GEMM: activations
    a [E, max_m, K] ~ N(0, 1) quantised per row and 128 columns, weights
    b [E, N, K] ~ N(0, 1/sqrt(K)) quantised per 128 x 128 block, and valid row
    counts uniform in [max_m/2, max_m] unless given.  Drawn on ``device`` one
    expert at a time."""
    g = torch.Generator(device=device)
    g.manual_seed(7_000_000 + seed)
    a = torch.empty((E, max_m, K), dtype=torch.float8_e4m3fn, device=device)
    b = torch.empty((E, N, K), dtype=torch.float8_e4m3fn, device=device)
    a_scale = torch.empty((E, max_m, K // 128), dtype=torch.float32, device=device)
    b_scale = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=device)
    for e in range(E):
        xa = torch.randn((max_m, K), generator=g, device=device, dtype=torch.float32)
        a[e], a_scale[e] = _quantize_blocks(xa, 1)
        xb = torch.randn((N, K), generator=g, device=device, dtype=torch.float32) / math.sqrt(K)
        b[e], b_scale[e] = _quantize_blocks(xb, 128)
    if counts is None:
        gc = torch.Generator()
        gc.manual_seed(7_100_000 + seed)
        counts = torch.randint(max_m // 2, max_m + 1, (E,), generator=gc, dtype=torch.int32)
    counts = torch.as_tensor(counts, dtype=torch.int32).to(device)
    return {"a": a, "a_scale": a_scale, "b": b, "b_scale": b_scale, "counts": counts}


def subset_tokens(T: int, n: int = 256) -> list:
    """Fixed token subset t_i = floor(i * T / n), i < n (all tokens when T <= n)."""
    if T <= n:
        return list(range(T))
    return [(i * T) // n for i in range(n)]
