"""Plain, slow, CPU oracle of the routed Mixture-of-Experts FFN forward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or call
this module.  It shares no code with the CUDA path: no kernels, headers,
helpers or constants.  Inputs are numpy arrays holding exactly the values the
GPU receives (bf16 and fp32 inputs convert to float64 without rounding).

Arithmetic is float64, except where the pages fix the precision:
scoring and selection of the router run in float32 ("Scoring and selection
run in float32 whatever the logits dtype" -- TileOPs "MoE Operators",
FusedTopKFwdOp), so the integer decisions (which experts are chosen) are taken
in float32 here as on the GPU.  Intermediate results are rounded to the operand
dtype exactly where the pages put a cast:

* the gated activation is rounded to the operand dtype before the down GEMM
  (TileOPs "MoE Operators", MoEGroupedGemmFwdOp: output written in the operand
  dtype; SharedExpertMLPFwdOp: "rounded to the input dtype before the down
  projection"),
* the down GEMM result (bias included) is rounded to the operand dtype
  (MoEExpertMLPFwdOp: b_down added "before its cast"),
* the weighted reduction over k accumulates unrounded and is cast once
  (MoEPostPermuteFwdOp: "apply routing weights, reduce top-k, and cast").

``round_mode=None`` skips those casts, for error-budget diagnostics.

Sources (page title, section):
  [MoERouter]  ONNX Runtime PR #32126 "[CUDA] Add MoERouter and SwiGLU contrib
               operators", sections MoERouter and SwiGLU.
  [ORT-MoE]    onnx-light-cpu "MoE (CPU)", LightOpSchema (inputs, attributes).
  [ORT-spec]   ONNX Runtime PR #25619 "Update MoE and qMoE spec", sections
               "SwiGLU Activation Function" and "Fusion Behavior".
  [TileOPs]    TileOPs "MoE Operators", one section per op.

Parity pins: every public function here is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, brute force and the worked values under
``tests/golden/``.
"""
from __future__ import annotations

import itertools
import math
from typing import Optional

import numpy as np

# [MoERouter] router_probs of an expert that is not chosen: -1e30, except in
# float16, whose largest finite magnitude (65504) it exceeds; there -1e4
NEG_SENTINEL_F32 = -1e30
NEG_SENTINEL_F16 = -1e4

ACT_SILU_AND_MUL = 0
ACT_SWIGLU = 1
ACT_IDENTITY = 2
ACT_GELU_AND_MUL = 3   # gated, stacked [TileOPs MoEGroupedGemmFwdOp]
ACT_RELU = 4           # non-gated [ORT-MoE activation_type]
ACT_GELU = 5
ACT_SILU = 6
GATED_ACTS = (ACT_SILU_AND_MUL, ACT_SWIGLU, ACT_GELU_AND_MUL)


# --------------------------------------------------------------------------
# rounding to the operand dtype
# --------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), returned as
    float64.  bfloat16 keeps 8 significant bits and float32's exponent range:
    a value m * 2**e (0.5 <= |m| < 1) is quantised to a multiple of 2**(e - 8),
    the exponent clamped at the subnormal floor 2**-133; results of 2**128 or
    more overflow to infinity."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0)
    xf = x[finite]
    _, e = np.frexp(xf)
    e = np.maximum(e, -125)  # below 2**-126 the quantum stays 2**-133
    q = np.ldexp(1.0, e - 8)
    r = np.rint(xf / q) * q  # rint rounds half to even
    r[np.abs(r) >= 2.0 ** 128] = np.inf * np.sign(r[np.abs(r) >= 2.0 ** 128])
    out[finite] = r
    return out


def round_to(x, dtype: Optional[str]) -> np.ndarray:
    """Cast to the operand dtype and back to float64; ``None`` leaves x as is."""
    x = np.asarray(x, dtype=np.float64)
    if dtype is None:
        return x
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f16":  # IEEE binary16, round to nearest even
        return x.astype(np.float16).astype(np.float64)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# 1. routing  [TileOPs FusedTopKFwdOp / FusedMoEFwdOp], [MoERouter]
# --------------------------------------------------------------------------
def expert_scores(logits, scoring: str, score_dtype=np.float32) -> np.ndarray:
    """Per-token expert scores.  softmax: s_e = exp(z_e - max z) / sum exp(z - max z);
    sigmoid: s_e = 1 / (1 + exp(-z_e)); sqrt_softplus [MoERouter scoring]:
    s_e = sqrt(log(1 + exp(z_e))) (the name read literally).  Computed in
    ``score_dtype`` (float32 per [TileOPs FusedTopKFwdOp])."""
    z = np.asarray(logits).astype(score_dtype)
    if scoring == "softmax":
        zmax = z.max(axis=1, keepdims=True)
        ex = np.exp(z - zmax)
        return ex / ex.sum(axis=1, keepdims=True)
    if scoring == "sigmoid":
        one = score_dtype(1.0)
        return one / (one + np.exp(-z))
    if scoring == "sqrt_softplus":
        return np.sqrt(np.logaddexp(score_dtype(0.0), z))
    raise ValueError(scoring)


def selection_scores(scores, correction_bias=None) -> np.ndarray:
    """u_e = s_e + bias_e when a correction bias is passed: it steers the
    selection only [TileOPs FusedMoEFwdOp, FusedTopKFwdOp init].  The pages
    leave NaN open; the reading taken: a NaN selection score ranks below every
    number (u = -inf), so it never displaces a finite score, in a group score
    or in the top-K."""
    if correction_bias is None:
        u = np.array(scores, copy=True)
    else:
        u = scores + np.asarray(correction_bias).astype(scores.dtype)[None, :]
    return np.where(np.isnan(u), -np.inf, u).astype(u.dtype)


def group_scores(u, G: int, biased: bool) -> np.ndarray:
    """[T, G] group scores: experts split into G groups of E/G consecutive
    experts; a group scores the sum of its two best biased scores when a
    correction bias is passed, its best score otherwise [TileOPs FusedTopKFwdOp]."""
    T, E = u.shape
    S = E // G
    srt = np.sort(u.reshape(T, G, S), axis=2)
    if biased:
        return srt[:, :, -1] + srt[:, :, -2]
    return srt[:, :, -1]


def restrict_to_groups(u, G: int, TG: int, biased: bool) -> np.ndarray:
    """Keep the TG best groups (ties to the lower group index); every expert of
    another group gets -inf [TileOPs FusedTopKFwdOp, "as vLLM's grouped_topk"]."""
    T, E = u.shape
    if G <= 1:
        return u
    gs = group_scores(u, G, biased)
    order = np.argsort(-gs, axis=1, kind="stable")  # stable: equal scores keep lower g first
    keep = np.zeros((T, G), dtype=bool)
    keep[np.arange(T)[:, None], order[:, :TG]] = True
    allowed = np.repeat(keep, E // G, axis=1)
    return np.where(allowed, u, -np.inf).astype(u.dtype)


def topk_ascending(u, K: int) -> np.ndarray:
    """The K largest selection scores, ties to the lower expert index
    [MoERouter: "Ties go to the lower expert index"], returned in ascending
    expert order (the pages leave the order of ids within a row open)."""
    order = np.argsort(-u, axis=1, kind="stable")
    return np.sort(order[:, :K], axis=1).astype(np.int32)


def route(logits, K: int, scoring: str = "softmax", renormalize: bool = True,
          G: int = 1, TG: int = 1, rsf: float = 1.0, correction_bias=None,
          expert_ids=None, local_start: int = 0, local_count: int = 0,
          route_scale: float = 1.0, score_dtype=np.float32,
          probs_dtype: Optional[str] = None) -> dict:
    """Router of one layer.

    Returns ``topk_ids`` [T,K] int32, ``topk_weights`` [T,K] float64 and, when
    ``local_count > 0``, the MoERouter outputs ``router_probs`` [T, local_count]
    and ``weight_scale`` [T].

    Steps [TileOPs FusedTopKFwdOp, FusedMoEFwdOp; MoERouter]:
      1. scores s (softmax or sigmoid), in float32;
      2. selection scores u = s + correction_bias (selection only);
      3. with G > 1, restrict to the TG best groups;
      4. top-K of u, ties to the lower index -- or, when ``expert_ids`` is given,
         those ids in their given order, the bias ignored (hash routing);
      5. weights w_k = s[id_k] (unbiased), divided by their sum when
         ``renormalize``, then times ``rsf`` once;
      6. MoERouter: w^_k = s[id_k] / sum_j s[id_j] (always normalised, no rsf);
         router_probs[t, j] = log(sum of w^ over routes on expert local_start+j)
         when that expert is chosen, -1e30 otherwise; weight_scale[t] =
         route_scale * (sum of w^ over local routes), 0 when none is local.
         ``probs_dtype`` (the MoERouter tensor type of router_probs): the logs
         rounded to it, and the sentinel -1e4 in "f16" (-1e30 rounded to it
         otherwise); None keeps float64 values and -1e30.
    """
    s = expert_scores(logits, scoring, score_dtype)
    T, E = s.shape
    if expert_ids is not None:
        ids = np.asarray(expert_ids, dtype=np.int32).reshape(T, K)
    else:
        u = selection_scores(s, correction_bias)
        u = restrict_to_groups(u, G, TG, correction_bias is not None)
        ids = topk_ascending(u, K)
    chosen = np.take_along_axis(s, ids.astype(np.int64), axis=1).astype(np.float64)
    w = chosen.copy()
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    w = w * float(rsf)
    out = {"topk_ids": ids, "topk_weights": w}
    if local_count > 0:
        wn = chosen / chosen.sum(axis=1, keepdims=True)
        sentinel = NEG_SENTINEL_F16 if probs_dtype == "f16" else NEG_SENTINEL_F32
        probs = np.full((T, local_count), sentinel, dtype=np.float64)
        scale = np.zeros(T, dtype=np.float64)
        for t in range(T):
            acc = {}
            for k in range(K):
                j = int(ids[t, k]) - local_start
                if 0 <= j < local_count:
                    acc[j] = acc.get(j, 0.0) + wn[t, k]
            for j, v in acc.items():
                probs[t, j] = math.log(v)
            scale[t] = route_scale * sum(acc.values()) if acc else 0.0
        out["router_probs"] = round_to(probs, probs_dtype)
        out["weight_scale"] = scale
    return out


def selection_margins(logits, K: int, scoring: str = "softmax", G: int = 1, TG: int = 1,
                      correction_bias=None, score_dtype=np.float64) -> np.ndarray:
    """Per-token distance of the routing decision from a tie: the smallest of
    (K-th minus (K+1)-th allowed selection score) and, with groups,
    (TG-th minus (TG+1)-th group score).  Used by the tests to redraw input
    rows whose decision a few ulp could flip."""
    s = expert_scores(logits, scoring, score_dtype)
    T, E = s.shape
    u = selection_scores(s, correction_bias)
    m = np.full(T, np.inf)
    if G > 1:
        gs = np.sort(group_scores(u, G, correction_bias is not None), axis=1)[:, ::-1]
        if TG < G:
            m = np.minimum(m, gs[:, TG - 1] - gs[:, TG])
        u = restrict_to_groups(u, G, TG, correction_bias is not None)
    us = np.sort(u, axis=1)[:, ::-1]
    if K < E:
        nxt = us[:, K]
        gap = np.where(np.isfinite(nxt), us[:, K - 1] - nxt, np.inf)
        m = np.minimum(m, gap)
    return m


# --------------------------------------------------------------------------
# 2. permutation into the tight expert-contiguous layout
#    [TileOPs MoEPrePermuteFwdOp; MoEGroupedGemmFwdOp "contiguous · physical_psum"]
# --------------------------------------------------------------------------
def permute(topk_ids, E: int) -> dict:
    """Route r = t*K + k goes to expert topk_ids[t,k].  counts[e] = routes on e;
    seg_end = inclusive prefix sum of counts (the segment END rows of the
    physical_psum layout).  Rows of expert e hold its routes in ascending r
    (the pages leave the order inside a segment open).  row_to_route[row] = r,
    route_to_row[r] = row."""
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    M = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    seg_end = np.cumsum(counts).astype(np.int32)
    row_to_route = np.argsort(flat, kind="stable").astype(np.int32)
    route_to_row = np.empty(M, dtype=np.int32)
    route_to_row[row_to_route] = np.arange(M, dtype=np.int32)
    return {"counts": counts.astype(np.int32), "seg_end": seg_end,
            "row_to_route": row_to_route, "route_to_row": route_to_row}


def permute_align(topk_ids, E: int, block_size: int) -> dict:
    """The padded layout of MoEPermuteAlignFwdOp [TileOPs "MoE Operators"]:
    with numel = T*K routes and count[e] of them on expert e,
    num_tokens_post_pad = sum over e of count[e] rounded up to block_size;
    sorted_token_ids (length numel + (E + 1) * (block_size - 1)) holds one range
    per expert, in expert order, of that rounded-up length, whose first count[e]
    slots are the routes on e (ascending route index here: the pages leave the
    order open) and the rest numel; every entry past num_tokens_post_pad is
    numel.  expert_ids (one per block_size block of sorted_token_ids) names
    the owner of each block of the ranges and is -1 past them."""
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    numel = flat.size
    L = numel + (E + 1) * (block_size - 1)
    sorted_ids = np.full(L, numel, dtype=np.int32)
    expert_ids = np.full(-(-L // block_size), -1, dtype=np.int32)
    pos = 0
    for e in range(E):
        routes = np.nonzero(flat == e)[0]
        padded = -(-len(routes) // block_size) * block_size
        sorted_ids[pos:pos + len(routes)] = routes
        expert_ids[pos // block_size:(pos + padded) // block_size] = e
        pos += padded
    return {"sorted_token_ids": sorted_ids, "expert_ids": expert_ids,
            "num_tokens_post_pad": np.int32(pos)}


def gather_rows(hidden, row_to_route, K: int) -> np.ndarray:
    """expert_input[row] = hidden[row_to_route[row] // K]."""
    h = np.asarray(hidden, dtype=np.float64)
    return h[np.asarray(row_to_route, dtype=np.int64) // K]


# --------------------------------------------------------------------------
# 3. activations  [ORT-spec SwiGLU; MoERouter SwiGLU; TileOPs MoEGroupedGemmFwdOp]
# --------------------------------------------------------------------------
def sigmoid64(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, dtype=np.float64)))


def gelu64(x):
    """GELU x * Phi(x) = x/2 * (1 + erf(x / sqrt(2))), the exact (erf) form:
    the pages name the activation without an approximation."""
    from scipy.special import erf

    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def swiglu_math(g, l, limit: float, alpha: float, beta: float) -> np.ndarray:
    """G = min(g, limit); L = max(min(l, limit), -limit);
    out = G * sigmoid(alpha * G) * (L + beta).  limit <= 0 disables both clamps
    [MoERouter SwiGLU; ORT-spec "SwiGLU Activation Function"]."""
    g = np.asarray(g, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    if limit > 0:
        G = np.minimum(g, limit)
        L = np.maximum(np.minimum(l, limit), -limit)
    else:
        G, L = g, l
    return G * sigmoid64(alpha * G) * (L + beta)


def split_gate_up(P, F: int, fusion: int):
    """Split the [.., 2F] gate/up product: fusion 1 interleaved (row 2j gate j,
    row 2j+1 up j), fusion 2 concatenated [g | l] (= the stacked gate rows then
    up rows of silu_and_mul) [ORT-spec "Fusion Behavior"; TileOPs
    MoEGroupedGemmFwdOp]."""
    P = np.asarray(P, dtype=np.float64)
    if fusion == 1:
        return P[..., 0:2 * F:2], P[..., 1:2 * F:2]
    if fusion == 2:
        return P[..., :F], P[..., F:2 * F]
    raise ValueError(f"swiglu_fusion {fusion}")


def gated_activation(P, F: int, act: int, fusion: int = 2, limit: float = 0.0,
                     alpha: float = 1.0, beta: float = 0.0) -> np.ndarray:
    """act(P) for the gate_up product P [.., 2F] (or [.., F] for identity).

    silu_and_mul: stacked, silu(gate) * up with silu(x) = x * sigmoid(x)
    [TileOPs MoEGroupedGemmFwdOp].  SWIGLU: the clamped SwiGLU over the layout
    ``fusion`` picks.  IDENTITY: the non-gated identity of [ORT-MoE]
    activation_type (used as a special case only)."""
    if act == ACT_SILU_AND_MUL:
        g, u = split_gate_up(P, F, 2)
        return g * sigmoid64(g) * u
    if act == ACT_GELU_AND_MUL:
        g, u = split_gate_up(P, F, 2)
        return gelu64(g) * u
    if act == ACT_SWIGLU:
        g, l = split_gate_up(P, F, fusion)
        return swiglu_math(g, l, limit, alpha, beta)
    p = np.asarray(P, dtype=np.float64)[..., :F]
    if act == ACT_IDENTITY:
        return p
    if act == ACT_RELU:
        return np.maximum(p, 0.0)
    if act == ACT_GELU:
        return gelu64(p)
    if act == ACT_SILU:
        return p * sigmoid64(p)
    raise ValueError(act)


def swiglu_op(gate, up, inter: int, fusion: int, limit: float, alpha: float, beta: float,
              dtype: Optional[str]) -> np.ndarray:
    """The standalone SwiGLU operator [MoERouter, section SwiGLU]: with ``up``
    given, gate and up are [R, inter]; without it ``gate`` is one [R, 2*inter]
    projection split per ``fusion`` (2: gate first then up; 1: interleaved).
    Output rounded to ``dtype``."""
    if up is None:
        g, l = split_gate_up(gate, inter, fusion)
    else:
        g, l = np.asarray(gate, np.float64), np.asarray(up, np.float64)
    return round_to(swiglu_math(g, l, limit, alpha, beta), dtype)


# --------------------------------------------------------------------------
# 4. expert GEMMs  [TileOPs MoEGroupedGemmFwdOp, MoEExpertMLPFwdOp]
# --------------------------------------------------------------------------
def _segments(seg_end):
    start = 0
    for e, end in enumerate(np.asarray(seg_end, dtype=np.int64)):
        yield e, start, int(end)
        start = int(end)


def grouped_gemm(a, b, seg_end, bias=None) -> np.ndarray:
    """Plain M-grouped NT GEMM on the physical_psum layout: for each expert g,
    out[rows of g] = a[rows of g] @ b[g]^T (+ bias[g]), in float64.
    a [M, K], b [E, N, K], bias [E, N]."""
    a = np.asarray(a, dtype=np.float64)
    M = a.shape[0]
    E, N, _ = b.shape
    out = np.zeros((M, N), dtype=np.float64)
    for e, s, t in _segments(seg_end):
        if t <= s:
            continue
        w = np.asarray(b[e], dtype=np.float64)
        out[s:t] = a[s:t] @ w.T
        if bias is not None:
            out[s:t] += np.asarray(bias[e], dtype=np.float64)[None, :]
    return out


def grouped_gemm_act(a, w_gate_up, seg_end, F: int, act: int, fusion: int = 2,
                     limit: float = 0.0, alpha: float = 1.0, beta: float = 0.0,
                     b_gate_up=None, dtype: Optional[str] = "bf16") -> np.ndarray:
    """gate_up GEMM with the gated activation fused: act(a @ W1[g]^T + b1[g]),
    bias added to the product before the activation and the cast, result cast
    to the operand dtype [TileOPs MoEGroupedGemmFwdOp]."""
    P = grouped_gemm(a, w_gate_up, seg_end, b_gate_up)
    return round_to(gated_activation(P, F, act, fusion, limit, alpha, beta), dtype)


def grouped_gemm_act_split(a, w_gate, w_up, seg_end, act: int, limit: float = 0.0,
                           alpha: float = 1.0, beta: float = 0.0, b_gate=None, b_up=None,
                           dtype: Optional[str] = "bf16") -> np.ndarray:
    """The gated gate_up GEMM with the gate and up projections in two weight
    tensors [ORT-spec "Fusion Behavior": swiglu_fusion 0, "two GEMMs are
    computed independently", FC1 giving g and FC3 giving l]: g = a @ Wg[e]^T
    (+ bg[e]), l = a @ Wu[e]^T (+ bu[e]), out = act(g, l) cast to ``dtype``,
    for act silu_and_mul, gelu_and_mul or the clamped SwiGLU."""
    g = grouped_gemm(a, w_gate, seg_end, b_gate)
    l = grouped_gemm(a, w_up, seg_end, b_up)
    F = g.shape[1]
    return round_to(gated_activation(np.concatenate([g, l], axis=1), F, act, 2, limit, alpha,
                                     beta), dtype)


def grouped_gemm_layout(a, b, layout: str, meta, act: Optional[int] = None, F: int = 0,
                        fusion: int = 2, limit: float = 0.0, alpha: float = 1.0,
                        beta: float = 0.0, bias=None, dtype: Optional[str] = "bf16"):
    """MoEGroupedGemmFwdOp over its three row layouts [TileOPs "MoE
    Operators", MoEGroupedGemmFwdOp layout table]: "psum" (a [M, K], meta the
    segment END rows), "per_row" (a [M, K], meta [M] the expert of every row,
    rows grouped by expert in ascending order, as the layout requires), or
    "masked" (a [E, max_m, K], meta [E] valid rows per expert, read as
    min(max(m, 0), max_m); out [E, max_m, N] with the rows past the count NaN
    here, "unspecified" on the pages).  With ``act`` the gated or non-gated
    activation is fused as in grouped_gemm_act, else the plain product (+
    bias) cast to ``dtype``."""
    def run(rows, seg_end):
        if act is None:
            return round_to(grouped_gemm(rows, b, seg_end, bias), dtype)
        return grouped_gemm_act(rows, b, seg_end, F, act, fusion, limit, alpha, beta, bias, dtype)

    if layout == "psum":
        return run(a, meta)
    if layout == "per_row":
        ids = np.asarray(meta, dtype=np.int64)
        if ids.size and np.any(np.diff(ids) < 0):
            raise ValueError("per_row ids must be grouped in ascending expert order")
        E = np.asarray(b).shape[0]
        return run(a, np.cumsum(np.bincount(ids, minlength=E)))
    if layout == "masked":
        A = np.asarray(a, dtype=np.float64)
        E, max_m, _ = A.shape
        m = np.clip(np.asarray(meta, dtype=np.int64), 0, max_m)
        packed = np.concatenate([A[e, :m[e]] for e in range(E)])
        y = run(packed, np.cumsum(m))
        out = np.full((E, max_m, y.shape[1]), np.nan)
        pos = 0
        for e in range(E):
            out[e, :m[e]] = y[pos:pos + m[e]]
            pos += m[e]
        return out
    raise ValueError(layout)


def grouped_gemm_down(a, w_down, seg_end, b_down=None, dtype: Optional[str] = "bf16"):
    """down GEMM: a @ W2[g]^T + b2[g] in float64, cast to the operand dtype
    [TileOPs MoEExpertMLPFwdOp]."""
    return round_to(grouped_gemm(a, w_down, seg_end, b_down), dtype)


# --------------------------------------------------------------------------
# 5. unpermute + weighted combine  [TileOPs MoEPostPermuteFwdOp, FusedMoEExpertsFwdOp]
# --------------------------------------------------------------------------
def combine(expert_out, topk_weights, route_to_row, T: int, K: int, scale: float = 1.0,
            dtype: Optional[str] = "bf16") -> np.ndarray:
    """out[t] = scale * sum_{k=0..K-1} w[t,k] * Y[route_to_row[t*K+k]], summed
    in k order, cast once to ``dtype``."""
    Y = np.asarray(expert_out, dtype=np.float64)
    w = np.asarray(topk_weights, dtype=np.float64).reshape(T, K)
    r2r = np.asarray(route_to_row, dtype=np.int64).reshape(T, K)
    acc = np.zeros((T, Y.shape[1]), dtype=np.float64)
    for k in range(K):
        acc += w[:, k:k + 1] * Y[r2r[:, k]]
    return round_to(scale * acc, dtype)


# --------------------------------------------------------------------------
# 6. the whole forward, per token  [TileOPs FusedMoEExpertsFwdOp, FusedMoEFwdOp]
# --------------------------------------------------------------------------
def expert_mlp_routes(hidden_rows, experts, w_gate_up, w_down, F: int, act: int,
                      fusion: int = 2, limit: float = 0.0, alpha: float = 1.0,
                      beta: float = 0.0, b_gate_up=None, b_down=None,
                      dtype: Optional[str] = "bf16") -> np.ndarray:
    """y_r = round(round(act(x_r W1[e_r]^T + b1[e_r])) W2[e_r]^T + b2[e_r]) for
    each route r (row x_r of ``hidden_rows``, expert ``experts[r]``).  Each
    expert's weights are converted to float64 once and applied to all of its
    routes; every output row is still its own independent dot products."""
    X = np.asarray(hidden_rows, dtype=np.float64)
    experts = np.asarray(experts, dtype=np.int64)
    H = X.shape[1]
    Y = np.zeros((X.shape[0], H), dtype=np.float64)
    for e in np.unique(experts):
        rows = np.nonzero(experts == e)[0]
        W1 = np.asarray(w_gate_up[e], dtype=np.float64)
        W2 = np.asarray(w_down[e], dtype=np.float64)
        P = X[rows] @ W1.T
        if b_gate_up is not None:
            P += np.asarray(b_gate_up[e], dtype=np.float64)[None, :]
        A = round_to(gated_activation(P, F, act, fusion, limit, alpha, beta), dtype)
        y = A @ W2.T
        if b_down is not None:
            y += np.asarray(b_down[e], dtype=np.float64)[None, :]
        Y[rows] = round_to(y, dtype)
    return Y


def ffn_forward(hidden, logits, w_gate_up, w_down, K: int, F: int, scoring="softmax",
                renormalize=True, G=1, TG=1, rsf=1.0, correction_bias=None, expert_ids=None,
                act=ACT_SILU_AND_MUL, fusion=2, limit=0.0, alpha=1.0, beta=0.0,
                b_gate_up=None, b_down=None, dtype: Optional[str] = "bf16",
                local_start=0, local_count=0, route_scale=1.0, tokens=None) -> dict:
    """Routed MoE FFN forward for the tokens ``tokens`` (all when None):
    out[t] = sum_k w[t,k] * (down_k(act(gate_up_k(h[t]) + b1_k)) + b2_k), with
    rsf folded into w once by the router [TileOPs FusedMoEExpertsFwdOp,
    FusedMoEFwdOp].  Returns the routing outputs and ``out`` (rounded to
    ``dtype``) plus ``out_unrounded`` (the float64 sum before the final cast)."""
    logits = np.asarray(logits)
    T = logits.shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    ids_in = None if expert_ids is None else np.asarray(expert_ids)[tok]
    r = route(logits[tok], K, scoring, renormalize, G, TG, rsf, correction_bias, ids_in,
              local_start, local_count, route_scale)
    ids, w = r["topk_ids"], r["topk_weights"]
    X = np.asarray(hidden, dtype=np.float64)[tok]
    n = len(tok)
    Xr = np.repeat(X, K, axis=0)  # route (i, k) -> row i*K + k
    Y = expert_mlp_routes(Xr, ids.reshape(-1), w_gate_up, w_down, F, act, fusion, limit,
                          alpha, beta, b_gate_up, b_down, dtype)
    acc = np.zeros((n, X.shape[1]), dtype=np.float64)
    for k in range(K):
        acc += w[:, k:k + 1] * Y[k::K]
    r["out_unrounded"] = acc
    r["out"] = round_to(acc, dtype)
    r["route_out"] = Y  # y of route (i, k) at row i*K + k, rounded to dtype
    r["tokens"] = tok
    return r


def ffn_forward_local(hidden, router_probs, weight_scale, w_gate_up, w_down, K: int, F: int,
                      act=ACT_SILU_AND_MUL, fusion=2, limit=0.0, alpha=1.0, beta=0.0,
                      dtype: Optional[str] = "bf16", parts: bool = False):
    """The layer of one expert-parallel rank holding lc experts (w_gate_up and
    w_down of those experts only), fed by the MoERouter outputs of its slice
    [MoERouter: "QMoE's own softmax over the local block returns w_e /
    W_local", "weight_scale ... multiplies that factor back out of the expert
    output before the all-reduce"]: the softmax of the token's router_probs
    row (float32, as the router computes it), its top min(K, lc) experts (ties
    to the lower index), the weighted sum of their expert MLPs, multiplied by
    weight_scale[t] and cast once.  Summed over the ranks' slices this is the
    routed layer with normalised weights (times route_scale).  ``parts``:
    return a dict with ``out``, ``out_unrounded`` (before the cast),
    ``route_out`` and ``topk_weights`` instead of the output alone."""
    rp = np.asarray(router_probs, dtype=np.float32)
    lc = rp.shape[1]
    Kl = min(K, lc)
    r = route(rp, Kl, "softmax", renormalize=False)
    X = np.asarray(hidden, dtype=np.float64)
    Xr = np.repeat(X, Kl, axis=0)
    Y = expert_mlp_routes(Xr, r["topk_ids"].reshape(-1), w_gate_up, w_down, F, act, fusion,
                          limit, alpha, beta, None, None, dtype)
    acc = np.zeros_like(X)
    for k in range(Kl):
        acc += r["topk_weights"][:, k:k + 1] * Y[k::Kl]
    exact = np.asarray(weight_scale, dtype=np.float64)[:, None] * acc
    if parts:
        return {"out": round_to(exact, dtype), "out_unrounded": exact, "route_out": Y,
                "topk_weights": r["topk_weights"]}
    return round_to(exact, dtype)


def shared_expert_mlp(hidden, w_gate_up, w_down, dtype: Optional[str] = "bf16",
                      unrounded: bool = False) -> np.ndarray:
    """Dense gated MLP of the shared expert, applied to every token
    [TileOPs SharedExpertMLPFwdOp]: with w_gate_up [2S, H] the gate rows (0..S)
    stacked over the up rows (S..2S) and w_down [H, S],
        out = down(silu(hidden @ gate^T) * (hidden @ up^T)),
    both products accumulated in float64 here (float32 on the GPU), the gated
    activation rounded to the input dtype before the down projection, the
    result rounded to it too (``unrounded``: the down product before that
    last cast)."""
    X = np.asarray(hidden, dtype=np.float64)
    Wgu = np.asarray(w_gate_up, dtype=np.float64)
    Wd = np.asarray(w_down, dtype=np.float64)
    S = Wgu.shape[0] // 2
    g = X @ Wgu[:S].T
    u = X @ Wgu[S:].T
    a = round_to(g * sigmoid64(g) * u, dtype)
    if unrounded:
        return a @ Wd.T
    return round_to(a @ Wd.T, dtype)


def ffn_forward_shared(hidden, logits, w_gate_up, w_down, shared_w_gate_up, shared_w_down,
                       dtype: Optional[str] = "bf16", **routed) -> dict:
    """Shared + routed MoE FFN [TileOPs FusedMoESharedExpertFwdOp]: the two
    outputs are returned apart, ``shared`` from shared_expert_mlp and the
    routed result of ffn_forward (routed_scaling_factor scales the routed
    output only, once, through the routing weights)."""
    r = ffn_forward(hidden, logits, w_gate_up, w_down, dtype=dtype, **routed)
    X = np.asarray(hidden)[r["tokens"]]
    r["shared_unrounded"] = shared_expert_mlp(X, shared_w_gate_up, shared_w_down, dtype,
                                              unrounded=True)
    r["shared"] = round_to(r["shared_unrounded"], dtype)
    return r


# --------------------------------------------------------------------------
# block-scaled FP8 grouped GEMM over a masked slab [TileOPs MoEGroupedGemmFP8FwdOp]
# --------------------------------------------------------------------------
def e4m3_to_float(codes) -> np.ndarray:
    """Values of float8_e4m3fn codes (uint8): 1 sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits; exponent 0 encodes subnormals m/8 * 2**-6; no
    infinities, and S.1111.111 (0x7F, 0xFF) is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


FP8_BLOCK = 128  # K (and N) block of one scale [TileOPs MoEGroupedGemmFP8FwdOp]


def grouped_gemm_fp8_masked(a_codes, a_scale, b_codes, b_scale, counts,
                            dtype: Optional[str] = "bf16") -> np.ndarray:
    """out[g, :m_g] = a[g, :m_g] @ b[g]^T with one float32 scale per row and
    128 K-columns of a (a_scale [E, max_m, K/128]) and one per 128 x 128 block
    of b (b_scale [E, N/128, K/128]): each 128-wide K block is contracted from
    the raw FP8 values, multiplied by its two scales and added to the
    accumulator; m_g = counts[g] read as min(max(m_g, 0), max_m).  Rows at or
    past m_g are undefined on the pages; NaN here.  Float64 arithmetic, the
    result rounded to ``dtype`` [TileOPs MoEGroupedGemmFP8FwdOp]."""
    A = e4m3_to_float(a_codes)
    B = e4m3_to_float(b_codes)
    sa = np.asarray(a_scale, dtype=np.float64)
    sb = np.asarray(b_scale, dtype=np.float64)
    E, max_m, K = A.shape
    N = B.shape[1]
    if K % FP8_BLOCK or N % FP8_BLOCK:
        raise ValueError("K and N must be multiples of 128")
    nkb = K // FP8_BLOCK
    out = np.full((E, max_m, N), np.nan)
    for g in range(E):
        m = min(max(int(counts[g]), 0), max_m)
        acc = np.zeros((m, N))
        for kb in range(nkb):
            ks = slice(kb * FP8_BLOCK, (kb + 1) * FP8_BLOCK)
            part = A[g, :m, ks] @ B[g, :, ks].T                     # raw FP8 values
            bs = np.repeat(sb[g, :, kb], FP8_BLOCK)[:N]             # b scale of each column
            acc += part * sa[g, :m, kb][:, None] * bs[None, :]
        out[g, :m] = round_to(acc, dtype)
    return out


# --------------------------------------------------------------------------
# brute force (tiny inputs only): used by the pins, never by the GPU tests
# --------------------------------------------------------------------------
def brute_force_selection(u_row, K: int, G: int, TG: int, biased: bool):
    """Enumerate every TG-subset of groups and every K-subset of the experts
    inside them; return (best group set, best expert set) by maximal total
    score, ties to the lexicographically smaller (lower-index) choice."""
    E = len(u_row)
    S = E // G
    groups = list(range(G))

    def gscore(g):
        vals = sorted(u_row[g * S:(g + 1) * S], reverse=True)
        return vals[0] + vals[1] if biased else vals[0]

    if G > 1:
        best_gs = None
        for comb in itertools.combinations(groups, TG):
            tot = sum(gscore(g) for g in comb)
            if best_gs is None or tot > best_gs[0]:
                best_gs = (tot, comb)
        allowed = [e for g in best_gs[1] for e in range(g * S, (g + 1) * S)]
        kept = best_gs[1]
    else:
        allowed = list(range(E))
        kept = (0,)
    best = None
    for comb in itertools.combinations(sorted(allowed), K):
        tot = sum(u_row[e] for e in comb)
        if best is None or tot > best[0]:
            best = (tot, comb)
    return kept, best[1]
