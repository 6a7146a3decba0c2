"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

None of these tests re-types the oracle's formulas: they check closed-form
points (tests/golden), invariants, special cases that reduce to a library
routine, and brute force on tiny inputs, chosen so that a dropped term, a wrong
sign or index, or a transposed operand in the oracle fails at least one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import cases
from mixture_experts_ffn_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


# ---------------------------------------------------------------- rounding
def test_round_bf16_matches_torch_on_float32_values():
    """bf16 rounding of float32 inputs reduces to torch's float32 -> bfloat16 cast."""
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),  # subnormal range
        (rng.standard_normal(2000) * 1e37).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38], dtype=np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1).
    assert O.round_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6.
    assert O.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    # just above halfway rounds up
    assert O.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7
    assert O.round_to(1.0 + 2.0 ** -30, "f32") == 1.0
    assert O.round_to(0.1, None) == 0.1


# ---------------------------------------------------------------- SwiGLU
def test_swiglu_golden_points():
    n = 0
    for line in _golden_lines("swiglu_points.txt"):
        vals = [float(v) for v in line.split("#")[0].split()]
        g, l, limit, alpha, beta, expected = vals
        got = O.swiglu_math(np.array([g]), np.array([l]), limit, alpha, beta)[0]
        assert got == pytest.approx(expected, rel=1e-14, abs=1e-15), line
        n += 1
    assert n >= 8


def test_swiglu_clamps():
    rng = np.random.default_rng(2)
    g = rng.standard_normal(1000) * 10
    l = rng.standard_normal(1000) * 10
    # limit <= 0 disables both clamps: same as a limit larger than every input
    for lim in (0.0, -1.0):
        np.testing.assert_array_equal(O.swiglu_math(g, l, lim, 1.702, 1.0),
                                      O.swiglu_math(g, l, 1e9, 1.702, 1.0))
    # clamping the inputs by hand, then running unclamped, is the clamped result
    gc = np.minimum(g, 7.0)
    lc = np.clip(l, -7.0, 7.0)
    np.testing.assert_allclose(O.swiglu_math(g, l, 7.0, 1.702, 1.0),
                               O.swiglu_math(gc, lc, 0.0, 1.702, 1.0), rtol=0, atol=0)
    # the gate is clamped from above only
    assert O.swiglu_math(np.array([-20.0]), np.array([1.0]), 7.0, 1.0, 0.0)[0] < 0


def test_swiglu_odd_part_identity():
    """With L + beta = 1: out(G) - out(-G) = G*s(aG) + G*s(-aG) = G, because
    sigmoid(x) + sigmoid(-x) = 1.  Fails if alpha or the sign of the sigmoid is
    misplaced."""
    G = np.linspace(-6, 6, 101)
    for alpha in (1.0, 1.702, 0.3):
        up = np.ones_like(G) * 0.75
        d = O.swiglu_math(G, up, 0.0, alpha, 0.25) - O.swiglu_math(-G, up, 0.0, alpha, 0.25)
        np.testing.assert_allclose(d, G, rtol=1e-13, atol=1e-13)


def test_silu_and_mul_layout_and_values():
    """silu_and_mul reads stacked gate rows then up rows: with gate = ln 3 and
    up = 2, silu(ln 3) * 2 = (3/4) ln 3 * 2; swapping the halves gives another value."""
    F = 3
    P = np.array([[math.log(3)] * F + [2.0] * F])
    out = O.gated_activation(P, F, O.ACT_SILU_AND_MUL)
    np.testing.assert_allclose(out, [[0.75 * math.log(3) * 2] * F], rtol=1e-14)
    # silu(0) = 0 whatever up is
    P0 = np.array([[0.0] * F + [123.0] * F])
    np.testing.assert_array_equal(O.gated_activation(P0, F, O.ACT_SILU_AND_MUL), np.zeros((1, F)))


def test_swiglu_fusion_layouts():
    """fusion 1 interleaves (gate, up) per column pair, fusion 2 concatenates."""
    F = 4
    g = np.array([[0.5, -1.0, 2.0, 0.0]])
    l = np.array([[1.0, 2.0, -3.0, 4.0]])
    inter = np.empty((1, 2 * F))
    inter[:, 0::2] = g
    inter[:, 1::2] = l
    cat = np.concatenate([g, l], axis=1)
    ref = O.swiglu_math(g, l, 7.0, 1.702, 1.0)
    np.testing.assert_array_equal(O.gated_activation(inter, F, O.ACT_SWIGLU, 1, 7.0, 1.702, 1.0), ref)
    np.testing.assert_array_equal(O.gated_activation(cat, F, O.ACT_SWIGLU, 2, 7.0, 1.702, 1.0), ref)
    # the op without `up` splits [gate | up] (fusion 2) exactly as with `up` given
    np.testing.assert_array_equal(O.swiglu_op(cat, None, F, 2, 7.0, 1.702, 1.0, None),
                                  O.swiglu_op(g, l, F, 2, 7.0, 1.702, 1.0, None))
    assert not np.allclose(O.gated_activation(inter, F, O.ACT_SWIGLU, 2, 7.0, 1.702, 1.0), ref)


# ---------------------------------------------------------------- routing
def _route_case(c):
    kw = dict(K=c["K"], scoring=c["scoring"], renormalize=c["renormalize"], G=c["G"],
              TG=c["TG"], rsf=c["rsf"])
    bias = None if c["bias"] is None else np.array(c["bias"], dtype=np.float32)
    return O.route(np.array(c["logits"], dtype=np.float32), correction_bias=bias,
                   local_start=c.get("local_start", 0), local_count=c.get("local_count", 0),
                   route_scale=c.get("route_scale", 1.0), **kw)


def test_routing_golden_cases():
    n = 0
    for line in _golden_lines("routing_cases.txt"):
        c = json.loads(line)
        r = _route_case(c)
        np.testing.assert_array_equal(r["topk_ids"], np.array(c["ids"]), err_msg=c["name"])
        np.testing.assert_allclose(r["topk_weights"], np.array(c["weights"]), rtol=1e-7,
                                   err_msg=c["name"])
        if "router_probs" in c:
            np.testing.assert_allclose(r["router_probs"], np.array(c["router_probs"]), rtol=1e-7,
                                       err_msg=c["name"])
            np.testing.assert_allclose(r["weight_scale"], np.array(c["weight_scale"]), rtol=1e-7)
        n += 1
    assert n >= 10


def test_scores_special_values():
    # sigmoid(0) = 1/2; softmax of equal logits = 1/E; softmax of logs = normalised values
    s = O.expert_scores(np.zeros((1, 4), np.float32), "sigmoid")
    np.testing.assert_array_equal(s, np.full((1, 4), 0.5, np.float32))
    s = O.expert_scores(np.zeros((1, 5), np.float32), "softmax")
    np.testing.assert_allclose(s, np.full((1, 5), 0.2), rtol=1e-7)
    v = np.array([1.0, 2.0, 3.0, 4.0])
    s = O.expert_scores(np.log(v)[None, :].astype(np.float32), "softmax")
    np.testing.assert_allclose(s[0], v / v.sum(), rtol=1e-6)
    # softmax is shift invariant and works in float32 (the pages' precision)
    s2 = O.expert_scores((np.log(v) + 50.0)[None, :].astype(np.float32), "softmax")
    assert s2.dtype == np.float32
    np.testing.assert_allclose(s2[0], v / v.sum(), rtol=1e-5)


def test_renormalised_weights_sum_and_subset_softmax():
    """Renormalised softmax weights of the chosen experts equal the softmax over
    the chosen logits alone; they sum to 1 (times rsf)."""
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=64)
    z = cases.guarded_logits(cfg).numpy()
    for rsf in (1.0, 2.5):
        r = O.route(z, 8, "softmax", True, rsf=rsf)
        np.testing.assert_allclose(r["topk_weights"].sum(1), rsf, rtol=1e-12)
        for t in range(z.shape[0]):
            sel = z[t, r["topk_ids"][t]].astype(np.float64)
            ex = np.array([math.exp(v - sel.max()) for v in sel])
            np.testing.assert_allclose(r["topk_weights"][t], rsf * ex / ex.sum(), rtol=2e-6)
    # without renormalise the weights are the plain scores (rsf still applied once)
    r = O.route(z, 8, "softmax", False, rsf=2.0)
    assert np.all(r["topk_weights"].sum(1) < 2.0)


def test_topk_is_the_k_largest_brute_force():
    """Brute force over every K-subset (and TG-subset of groups) on tiny inputs:
    the chosen groups maximise the total group score, the chosen experts the
    total selection score, ties to the lower index."""
    rng = np.random.default_rng(3)
    for E, G_list in ((8, (1, 2, 4)), (6, (1, 2, 3)), (10, (1, 2, 5))):
        for G in G_list:
            S = E // G
            for TG in range(1, G + 1):
                for K in range(1, min(TG * S, 4) + 1):
                    for trial in range(6):
                        # dyadic values keep float32 sums exact; small range forces ties
                        z = (rng.integers(-4, 5, size=(1, E)) / 4.0).astype(np.float32)
                        bias = (rng.integers(-2, 3, size=E) / 8.0).astype(np.float32) \
                            if trial % 2 else None
                        scoring = "sigmoid" if bias is not None else ("softmax" if trial % 3 else "sigmoid")
                        r = O.route(z, K, scoring, True, G=G, TG=TG, correction_bias=bias)
                        s = O.expert_scores(z, scoring)
                        u = (s + bias[None, :]) if bias is not None else s
                        _, best = O.brute_force_selection([float(x) for x in u[0]], K, G, TG,
                                                          bias is not None)
                        assert tuple(r["topk_ids"][0]) == tuple(best), (E, G, TG, K, z, bias)


def test_group_restriction_matters_and_ties_to_lower_group():
    # all experts equal: every group ties -> the TG lowest groups, then lowest experts
    z = np.zeros((1, 12), np.float32)
    b = np.zeros(12, np.float32)
    r = O.route(z, 3, "sigmoid", True, G=4, TG=2, correction_bias=b)
    assert list(r["topk_ids"][0]) == [0, 1, 2]
    # a single strong expert in an otherwise weak group is dropped with its group
    b = np.array([0, 0, 0, 0.5, -1, -1, 0.25, 0.25, 0], np.float32)
    r1 = O.route(np.zeros((1, 9), np.float32), 2, "sigmoid", True, G=1, correction_bias=b)
    r3 = O.route(np.zeros((1, 9), np.float32), 2, "sigmoid", True, G=3, TG=1, correction_bias=b)
    assert list(r1["topk_ids"][0]) == [3, 6]
    assert list(r3["topk_ids"][0]) == [6, 7]


def test_bias_steers_selection_only():
    """Weights are the unbiased scores of the chosen experts: forcing the same ids
    without a bias (hash routing) gives identical weights."""
    cfg = synth.CONFIGS["deepseek_v3_bf16"].replace(T=128)
    z = cases.guarded_logits(cfg).numpy()
    b = synth.make_correction_bias(cfg).numpy()
    r = O.route(z, 8, "sigmoid", True, G=8, TG=4, rsf=2.5, correction_bias=b)
    r2 = O.route(z, 8, "sigmoid", True, rsf=2.5, expert_ids=r["topk_ids"])
    np.testing.assert_array_equal(r["topk_weights"], r2["topk_weights"])
    # a constant bias shifts every score equally: neither ids nor weights change
    r3 = O.route(z, 8, "sigmoid", True, G=8, TG=4, rsf=2.5, correction_bias=b + np.float32(0.25))
    np.testing.assert_array_equal(r["topk_ids"], r3["topk_ids"])
    # no renormalise, rsf 1: the weights are exactly the float32 sigmoid scores
    r4 = O.route(z, 8, "sigmoid", False, correction_bias=b, G=8, TG=4)
    s = O.expert_scores(z, "sigmoid")
    np.testing.assert_array_equal(r4["topk_weights"], np.take_along_axis(s, r4["topk_ids"].astype(np.int64), 1))


def test_hash_routing_ignores_bias_and_keeps_order():
    cfg = synth.CONFIGS["kimi_k2_decode_bf16"].replace(hash_ids=True)
    ids = synth.make_expert_ids(cfg).numpy()
    z = synth.make_logits(cfg).numpy()
    b = synth.make_correction_bias(cfg).numpy()
    r1 = O.route(z, 8, "sigmoid", True, rsf=2.827, correction_bias=b, expert_ids=ids)
    r2 = O.route(z, 8, "sigmoid", True, rsf=2.827, correction_bias=None, expert_ids=ids)
    np.testing.assert_array_equal(r1["topk_ids"], ids)
    np.testing.assert_array_equal(r1["topk_weights"], r2["topk_weights"])
    assert all(len(set(row)) == 8 for row in ids)


def test_float32_and_float64_selection_agree_on_guarded_rows():
    for name in ("qwen3_bf16", "deepseek_v3_bf16", "gpt_oss_bf16"):
        cfg = synth.CONFIGS[name].replace(T=min(512, synth.CONFIGS[name].T))
        z = cases.guarded_logits(cfg).numpy()
        cb = synth.make_correction_bias(cfg)
        b = None if cb is None else cb.numpy()
        kw = dict(K=cfg.K, scoring=cfg.scoring, G=cfg.G, TG=cfg.TG, correction_bias=b)
        a = O.route(z, score_dtype=np.float32, **kw)["topk_ids"]
        c = O.route(z, score_dtype=np.float64, **kw)["topk_ids"]
        np.testing.assert_array_equal(a, c)
        assert O.selection_margins(z, cfg.K, cfg.scoring, cfg.G, cfg.TG, b).min() >= cases.MIN_GAP


def test_moerouter_qmoe_softmax_invariant():
    """QMoE applies its own softmax to the local block of router_probs; that
    softmax must return w_e / W_local on local chosen experts and 0 elsewhere,
    and sum over slices of weight_scale * softmax(row) recovers w (route_scale 1)."""
    from scipy.special import softmax

    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=256)
    z = cases.guarded_logits(cfg).numpy()
    E, K = cfg.E, cfg.K
    full = O.route(z, K, "softmax", True)
    w_hat = np.zeros((z.shape[0], E))
    for t in range(z.shape[0]):
        for k in range(K):
            w_hat[t, full["topk_ids"][t, k]] += full["topk_weights"][t, k]
    recon = np.zeros_like(w_hat)
    for start in range(0, E, 32):
        r = O.route(z, K, "softmax", True, local_start=start, local_count=32, route_scale=1.0)
        p, ws = r["router_probs"], r["weight_scale"]
        for t in range(z.shape[0]):
            local = w_hat[t, start:start + 32]
            if local.sum() == 0:
                assert ws[t] == 0.0 and np.all(p[t] == -1e30)
                continue
            sm = softmax(p[t])
            np.testing.assert_allclose(sm, local / local.sum(), rtol=1e-10, atol=1e-300)
            np.testing.assert_allclose(ws[t], local.sum(), rtol=1e-12)
            recon[t, start:start + 32] = ws[t] * sm
    np.testing.assert_allclose(recon, w_hat, rtol=1e-10, atol=1e-300)


def test_expert_parallel_slices_sum_to_the_layer():
    """The expert-parallel contract end to end: every rank runs its experts
    from its own MoERouter outputs (router_probs through its own softmax and
    top-k, the sum scaled by weight_scale); the ranks' outputs add up to the
    routed layer with normalised weights, on every token, including tokens
    with no expert on a rank."""
    rng = np.random.default_rng(31)
    T, H, F, E, K, lc = 40, 8, 4, 16, 4, 4
    x = O.round_bf16(rng.standard_normal((T, H)))
    z = rng.standard_normal((T, E)).astype(np.float32) * 2.0
    w_gu = O.round_bf16(rng.standard_normal((E, 2 * F, H)) * 0.3)
    w_d = O.round_bf16(rng.standard_normal((E, H, F)) * 0.3)
    full = O.ffn_forward(x, z, w_gu, w_d, K=K, F=F, renormalize=True, rsf=1.0, dtype=None)["out"]
    total = np.zeros_like(full)
    n_empty = 0
    for start in range(0, E, lc):
        r = O.route(z, K, "softmax", True, local_start=start, local_count=lc, route_scale=1.0)
        n_empty += int((r["weight_scale"] == 0).sum())
        total += O.ffn_forward_local(x, r["router_probs"], r["weight_scale"],
                                     w_gu[start:start + lc], w_d[start:start + lc], K, F,
                                     dtype=None)
    assert n_empty > 0  # some rank holds none of some token's experts
    np.testing.assert_allclose(total, full, rtol=2e-6, atol=2e-6 * np.abs(full).max())


def _f16_grid():
    """Every finite IEEE binary16 value, built from its fields (sign, 5-bit
    exponent with bias 15, 10-bit fraction; exponent 0 subnormal), ascending,
    with the parity of each value's fraction field."""
    val, par = [], []
    for f in range(1024):  # zero and the subnormals
        val.append(f * 2.0 ** -24)
        par.append(f & 1)
    for e in range(1, 31):
        for f in range(1024):
            val.append((1024 + f) * 2.0 ** (e - 25))
            par.append(f & 1)
    val, par = np.array(val), np.array(par)
    return np.concatenate([-val[:0:-1], val]), np.concatenate([par[:0:-1], par])


def test_f16_rounding_against_the_grid():
    """round_to(x, "f16") is the nearest binary16 value, ties to the even
    fraction, overflow to infinity at 65520 = 65504 + half its spacing."""
    grid, odd = _f16_grid()
    assert grid[-1] == 65504.0 and len(grid) == 2 * 31744 - 1
    rng = np.random.default_rng(17)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.uniform(-8, 4.8, 3000),
                        (grid[:-1] + grid[1:]) / 2])  # every midpoint: a tie
    x = x[np.abs(x) < 65504.0]
    got = O.round_to(x, "f16")
    for v, g in zip(x, got):
        j = np.searchsorted(grid, v)
        lo, hi = grid[j - 1], grid[j]
        want = lo if (v - lo < hi - v or (v - lo == hi - v and not odd[j - 1])) else hi
        assert g == want or (g == 0 and want == 0), (v, g, want)
    assert np.isinf(O.round_to(np.array([65520.0, -1e30]), "f16")).all()
    assert O.round_to(np.array([65519.99]), "f16")[0] == 65504.0


def test_moerouter_f16_sentinel_survives_and_keeps_the_invariant():
    """In float16 router_probs, -1e30 would overflow to -inf (a token with no
    local expert would give QMoE's softmax a row of -inf: NaN); the -1e4
    sentinel stays finite, that row's softmax is the degenerate uniform one
    (weight_scale 0 removes it), and on other rows the softmax over the f16
    logs still returns w_e / W_local to float16 precision and exactly 0 at
    the sentinel."""
    from scipy.special import softmax

    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=256)
    z = cases.guarded_logits(cfg).numpy()
    E, K, lc = cfg.E, cfg.K, 16
    assert np.isinf(O.round_to(np.array([O.NEG_SENTINEL_F32]), "f16")).all()
    n_empty = 0
    for start in range(0, E, lc):
        r = O.route(z, K, "softmax", True, local_start=start, local_count=lc, probs_dtype="f16")
        x = O.route(z, K, "softmax", True, local_start=start, local_count=lc)
        p = r["router_probs"]
        np.testing.assert_array_equal(p, O.round_to(p, "f16"))  # representable
        assert np.isfinite(p).all()
        for t in range(z.shape[0]):
            sm = softmax(p[t].astype(np.float32))
            assert np.isfinite(sm).all()
            if r["weight_scale"][t] == 0:
                n_empty += 1
                assert np.all(p[t] == -1e4)
                continue
            want = softmax(x["router_probs"][t])
            assert np.all(sm[want == 0] == 0)
            # |log w| <= ~12 here, so one f16 rounding of a log moves w by < 2^-11 * 12
            np.testing.assert_allclose(sm, want, rtol=8e-3, atol=0)
    assert n_empty > 0


def test_moerouter_normalises_even_without_renormalize():
    z = np.log(np.array([[1.0, 2.0, 3.0, 4.0]], np.float32))
    r = O.route(z, 2, "softmax", False, rsf=3.0, local_start=0, local_count=4)
    # chosen: experts 2, 3 with scores 3/10, 4/10; w^ = 3/7, 4/7, no rsf
    np.testing.assert_allclose(np.exp(r["router_probs"][0, 2:]), [3 / 7, 4 / 7], rtol=1e-6)
    assert np.all(r["router_probs"][0, :2] == -1e30)
    np.testing.assert_allclose(r["topk_weights"][0], [0.9, 1.2], rtol=1e-6)


# ---------------------------------------------------------------- permutation
def test_permute_brute_force_and_invariants():
    rng = np.random.default_rng(4)
    for T, K, E in ((1, 1, 1), (5, 2, 3), (17, 3, 8), (64, 4, 16), (33, 8, 8)):
        ids = np.stack([rng.choice(E, size=K, replace=K > E) for _ in range(T)]).astype(np.int32)
        p = O.permute(ids, E)
        flat = ids.reshape(-1)
        # brute force: walk experts in order, and routes in ascending order inside each
        rows = [r for e in range(E) for r in range(flat.size) if flat[r] == e]
        np.testing.assert_array_equal(p["row_to_route"], rows)
        counts = [sum(1 for v in flat if v == e) for e in range(E)]
        np.testing.assert_array_equal(p["counts"], counts)
        assert p["seg_end"][-1] == T * K
        np.testing.assert_array_equal(np.diff(np.concatenate([[0], p["seg_end"]])), counts)
        np.testing.assert_array_equal(p["route_to_row"][p["row_to_route"]], np.arange(T * K))
    # every route on one expert; empty experts in between
    ids = np.full((7, 2), 5, np.int32)
    p = O.permute(ids, 9)
    assert list(p["seg_end"]) == [0, 0, 0, 0, 0, 14, 14, 14, 14]


# ---------------------------------------------------------------- GEMMs
def _perm_matrix(n_out, n_in, shift, scale):
    """W[n, h] = scale if h == (n + shift) % n_in else 0."""
    W = np.zeros((n_out, n_in))
    for n in range(n_out):
        W[n, (n + shift) % n_in] = scale
    return W


def test_grouped_gemm_orientation_expert_and_bias():
    """Selection-matrix weights give closed forms: out[row, n] = c_e * a[row, (n + e) % K]
    + bias[e, n].  A transposed operand, a wrong expert or a dropped bias fails."""
    E, N, Kd = 3, 5, 7
    b = np.stack([_perm_matrix(N, Kd, e, float(e + 2)) for e in range(E)])
    bias = np.arange(E * N, dtype=np.float64).reshape(E, N) / 8.0
    seg_end = np.array([2, 2, 6])  # expert 1 empty
    rng = np.random.default_rng(5)
    a = rng.standard_normal((6, Kd))
    out = O.grouped_gemm(a, b, seg_end, bias)
    expert_of_row = [0, 0, 2, 2, 2, 2]
    for row in range(6):
        e = expert_of_row[row]
        for n in range(N):
            assert out[row, n] == pytest.approx((e + 2) * a[row, (n + e) % Kd] + bias[e, n], abs=1e-14)


def test_dense_reduction_identity_one_expert_brute_force():
    """E=1, K=1, identity activation, no rounding: the layer is the dense
    (x W1^T + b1) W2^T + b2 (times the weight 1).  Checked with explicit sums."""
    rng = np.random.default_rng(6)
    T, H, F = 4, 6, 3
    x = rng.standard_normal((T, H))
    W1 = rng.standard_normal((1, F, H))
    W2 = rng.standard_normal((1, H, F))
    b1 = rng.standard_normal((1, F))
    b2 = rng.standard_normal((1, H))
    r = O.ffn_forward(x, np.zeros((T, 1), np.float32), W1, W2, K=1, F=F, act=O.ACT_IDENTITY,
                      b_gate_up=b1, b_down=b2, dtype=None)
    for t in range(T):
        p = [sum(x[t, h] * W1[0, f, h] for h in range(H)) + b1[0, f] for f in range(F)]
        y = [sum(p[f] * W2[0, h, f] for f in range(F)) + b2[0, h] for h in range(H)]
        np.testing.assert_allclose(r["out"][t], y, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(r["topk_weights"], np.ones((T, 1)))


def test_staged_pipeline_equals_per_token_definition():
    """route -> permute -> grouped GEMMs -> combine gives the same result as the
    per-token formula (same rounding points), on a small bf16 and fp32 case."""
    for name, over in (("tiny_fp32", {}),
                       ("gpt_oss_bf16", dict(T=40, H=64, F=48, E=6, K=3)),
                       ("deepseek_v3_bf16", dict(T=40, H=64, F=32, E=16, K=4, G=4, TG=2))):
        cfg = synth.CONFIGS[name].replace(**over)
        inp = synth.make_inputs(cfg, "cpu", logits=cases.guarded_logits(cfg))
        n = {k: cases.to_np(v) for k, v in inp.items()}
        kw = dict(act=cfg.act, fusion=cfg.swiglu_fusion, limit=cfg.limit, alpha=cfg.alpha,
                  beta=cfg.beta)
        full = O.ffn_forward(n["hidden"], n["logits"], n["w_gate_up"], n["w_down"],
                             correction_bias=n["correction_bias"], b_gate_up=n["b_gate_up"],
                             b_down=n["b_down"], F=cfg.F, dtype=cfg.dtype,
                             **cases.oracle_kwargs(cfg), **kw)
        r = O.route(n["logits"], correction_bias=n["correction_bias"], **cases.oracle_kwargs(cfg))
        p = O.permute(r["topk_ids"], cfg.E)
        a = O.gather_rows(n["hidden"], p["row_to_route"], cfg.K)
        act = O.grouped_gemm_act(a, n["w_gate_up"], p["seg_end"], cfg.F, b_gate_up=n["b_gate_up"],
                                 dtype=cfg.dtype, **{k2: v for k2, v in kw.items()})
        y = O.grouped_gemm_down(act, n["w_down"], p["seg_end"], n["b_down"], cfg.dtype)
        out = O.combine(y, r["topk_weights"], p["route_to_row"], cfg.T, cfg.K, 1.0, cfg.dtype)
        np.testing.assert_allclose(out, full["out"], rtol=0, atol=1e-12)


def test_linearity_in_rsf_and_combine_one_hot():
    cfg = synth.CONFIGS["deepseek_v3_bf16"].replace(T=24, H=32, F=16, E=16, K=4, G=4, TG=2)
    inp = synth.make_inputs(cfg, "cpu", logits=cases.guarded_logits(cfg))
    n = {k: cases.to_np(v) for k, v in inp.items()}
    outs = {}
    for rsf in (1.0, 2.5):
        outs[rsf] = O.ffn_forward(n["hidden"], n["logits"], n["w_gate_up"], n["w_down"], K=4, F=16,
                                  scoring="sigmoid", G=4, TG=2, rsf=rsf,
                                  correction_bias=n["correction_bias"], dtype=None)["out"]
    np.testing.assert_allclose(outs[2.5], 2.5 * outs[1.0], rtol=1e-12, atol=1e-14)
    # combine with one-hot expert outputs places each weight at its row's column
    T, K, H = 3, 2, 6
    Y = np.eye(T * K, H)
    w = np.array([[0.25, 0.75], [1.0, 2.0], [-1.0, 0.5]])
    r2r = np.array([3, 0, 5, 1, 2, 4])
    out = O.combine(Y, w, r2r, T, K, scale=2.0, dtype=None)
    exp = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            exp[t, r2r[t * K + k]] += 2.0 * w[t, k]
    np.testing.assert_array_equal(out, exp)


def test_shared_expert_golden_points():
    """SharedExpertMLPFwdOp on the hand-derived points (no casts)."""
    L = math.log(3.0)
    w_gu = np.array([[L, 0.0], [0.0, L], [2.0, 7.0], [4.0, 1.0]])
    w_d = np.array([[1.0, 3.0], [-2.0, 5.0]])
    n = 0
    for line in _golden_lines("shared_expert_points.txt"):
        x0, x1, o0, o1 = (float(v) for v in line.split())
        out = O.shared_expert_mlp(np.array([[x0, x1]]), w_gu, w_d, dtype=None)
        np.testing.assert_allclose(out[0], [o0, o1], rtol=1e-13, atol=1e-13)
        n += 1
    assert n == 3


def test_shared_expert_brute_force_with_casts():
    """The shared expert against explicit loops over tokens, hidden and
    intermediate columns, with the casts where SharedExpertMLPFwdOp puts them
    (the gated activation rounded to the input dtype before the down GEMM,
    the result rounded too)."""
    rng = np.random.default_rng(11)
    T, H, S = 3, 5, 4
    x = O.round_bf16(rng.standard_normal((T, H)))
    w_gu = O.round_bf16(rng.standard_normal((2 * S, H)) * 0.5)
    w_d = O.round_bf16(rng.standard_normal((H, S)) * 0.5)
    want = np.zeros((T, H))
    for t in range(T):
        act = []
        for s in range(S):
            g = sum(x[t, h] * w_gu[s, h] for h in range(H))
            u = sum(x[t, h] * w_gu[S + s, h] for h in range(H))
            act.append(float(O.round_bf16(g / (1.0 + math.exp(-g)) * u)))
        for h in range(H):
            want[t, h] = float(O.round_bf16(sum(act[s] * w_d[h, s] for s in range(S))))
    np.testing.assert_array_equal(O.shared_expert_mlp(x, w_gu, w_d, dtype="bf16"), want)


def test_shared_plus_routed_returns_both_apart():
    """FusedMoESharedExpertFwdOp: the routed output is the routed forward's
    (rsf applied once, to it only) and the shared output the shared MLP's."""
    rng = np.random.default_rng(12)
    T, H, F, E, K, S = 6, 8, 4, 4, 2, 6
    x = O.round_bf16(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    w_gu = O.round_bf16(rng.standard_normal((E, 2 * F, H)) * 0.3)
    w_d = O.round_bf16(rng.standard_normal((E, H, F)) * 0.3)
    s_gu = O.round_bf16(rng.standard_normal((2 * S, H)) * 0.3)
    s_d = O.round_bf16(rng.standard_normal((H, S)) * 0.3)
    r1 = O.ffn_forward_shared(x, logits, w_gu, w_d, s_gu, s_d, dtype=None, K=K, F=F, rsf=1.0)
    r3 = O.ffn_forward_shared(x, logits, w_gu, w_d, s_gu, s_d, dtype=None, K=K, F=F, rsf=3.0)
    np.testing.assert_allclose(r3["out"], 3.0 * r1["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(r3["shared"], r1["shared"])
    np.testing.assert_array_equal(r1["shared"], O.shared_expert_mlp(x, s_gu, s_d, dtype=None))


def test_e4m3_golden_points():
    n = 0
    for line in _golden_lines("e4m3_points.txt"):
        code, val = line.split()[:2]
        got = float(O.e4m3_to_float(np.array([int(code, 16)], dtype=np.uint8))[0])
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val) and math.copysign(1.0, got) == math.copysign(1.0, float(val)), code
        n += 1
    assert n == 16


def test_e4m3_every_code_matches_torch():
    """Every code decodes as torch's own float8_e4m3fn conversion does."""
    codes = np.arange(256, dtype=np.uint8)
    mine = O.e4m3_to_float(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])


def _fp8_case(rng, E, max_m, N, K, int_values=False):
    if int_values:  # small integers: 1..4 and their negatives are exact e4m3 values
        lut = {1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48}
        va = rng.integers(-4, 5, size=(E, max_m, K))
        vb = rng.integers(-4, 5, size=(E, N, K))
        enc = np.vectorize(lambda v: 0 if v == 0 else (lut[abs(v)] | (0x80 if v < 0 else 0)))
        a, b = enc(va).astype(np.uint8), enc(vb).astype(np.uint8)
    else:
        a = rng.integers(0, 256, size=(E, max_m, K)).astype(np.uint8)
        b = rng.integers(0, 256, size=(E, N, K)).astype(np.uint8)
        a[(a & 0x7F) == 0x7F] = 0x38   # no NaN codes
        b[(b & 0x7F) == 0x7F] = 0x38
    sa = np.exp2(rng.integers(-3, 4, size=(E, max_m, K // 128))).astype(np.float32)
    sb = np.exp2(rng.integers(-3, 4, size=(E, N // 128, K // 128))).astype(np.float32)
    return a, sa, b, sb


def test_fp8_grouped_gemm_brute_force():
    """Block-scaled FP8 masked GEMM against explicit loops: per 128-wide K
    block the raw FP8 products are summed, then scaled by the row's and the
    block's scale [TileOPs MoEGroupedGemmFP8FwdOp]; rows past the count are
    left undefined."""
    rng = np.random.default_rng(21)
    E, max_m, N, K = 2, 3, 128, 256
    a, sa, b, sb = _fp8_case(rng, E, max_m, N, K, int_values=True)
    counts = [3, 2]
    got = O.grouped_gemm_fp8_masked(a, sa, b, sb, counts, dtype=None)
    va, vb = O.e4m3_to_float(a), O.e4m3_to_float(b)
    for g in range(E):
        for r in range(max_m):
            if r >= counts[g]:
                assert np.isnan(got[g, r]).all()
                continue
            for n in range(0, N, 37):
                total = 0.0
                for kb in range(K // 128):
                    part = sum(va[g, r, k] * vb[g, n, k] for k in range(kb * 128, kb * 128 + 128))
                    total += part * float(sa[g, r, kb]) * float(sb[g, n // 128, kb])
                assert got[g, r, n] == total, (g, r, n)


def test_fp8_scales_act_per_block():
    """Doubling one K block's scales doubles that block's contribution only."""
    rng = np.random.default_rng(22)
    E, max_m, N, K = 1, 4, 256, 384
    a, sa, b, sb = _fp8_case(rng, E, max_m, N, K)
    base = O.grouped_gemm_fp8_masked(a, sa, b, sb, [4], dtype=None)
    sa2 = sa.copy()
    sa2[:, :, 1] *= 2
    twice = O.grouped_gemm_fp8_masked(a, sa2, b, sb, [4], dtype=None)
    va, vb = O.e4m3_to_float(a), O.e4m3_to_float(b)
    blk = (va[0, :, 128:256] @ vb[0, :, 128:256].T) * sa[0, :, 1][:, None] * \
        np.repeat(sb[0, :, 1], 128)[None, :]
    np.testing.assert_allclose(twice[0] - base[0], blk, rtol=1e-12, atol=1e-9)
    sb2 = sb.copy()
    sb2[0, 1, 0] *= 4  # columns 128..255, K block 0
    other = O.grouped_gemm_fp8_masked(a, sa, b, sb2, [4], dtype=None)
    np.testing.assert_array_equal(other[0, :, :128], base[0, :, :128])
    assert not np.array_equal(other[0, :, 128:], base[0, :, 128:])


def test_fp8_counts_are_clamped():
    """A count past max_m is read as max_m, a negative one as 0."""
    rng = np.random.default_rng(23)
    a, sa, b, sb = _fp8_case(rng, 3, 5, 128, 128)
    got = O.grouped_gemm_fp8_masked(a, sa, b, sb, [-3, 99, 2], dtype=None)
    assert np.isnan(got[0]).all()
    assert not np.isnan(got[1]).any()
    full = O.grouped_gemm_fp8_masked(a, sa, b, sb, [5, 5, 5], dtype=None)
    np.testing.assert_array_equal(got[1], full[1])
    np.testing.assert_array_equal(got[2, :2], full[2, :2])


def test_activation_and_score_golden_points():
    kinds = {"relu": O.ACT_RELU, "gelu": O.ACT_GELU, "silu": O.ACT_SILU}
    n = 0
    for line in _golden_lines("activation_points.txt"):
        kind, a, b, want = line.split()[:4]
        a, b, want = float(a), float(b), float(want)
        if kind in kinds:
            got = O.gated_activation(np.array([[a]]), 1, kinds[kind])[0, 0]
        elif kind == "gelu_and_mul":
            got = O.gated_activation(np.array([[a, b]]), 1, O.ACT_GELU_AND_MUL)[0, 0]
        else:
            got = O.expert_scores(np.array([[a]]), "sqrt_softplus", np.float64)[0, 0]
        assert abs(got - want) <= 1e-15 * max(1.0, abs(want)), (kind, a, got, want)
        n += 1
    assert n == 12


def test_gelu_odd_part_and_stacked_layout():
    """gelu(x) - gelu(-x) = x (Phi(-x) = 1 - Phi(x)); gelu_and_mul takes the
    gate from the first F columns and the up from the last F."""
    x = np.linspace(-6, 6, 97)
    np.testing.assert_allclose(O.gelu64(x) - O.gelu64(-x), x, rtol=0, atol=1e-14)
    P = np.array([[1.0, 2.0, 3.0, 5.0]])
    np.testing.assert_allclose(O.gated_activation(P, 2, O.ACT_GELU_AND_MUL)[0],
                               [O.gelu64(1.0) * 3.0, O.gelu64(2.0) * 5.0], rtol=1e-15)


def test_sqrt_softplus_routes_like_any_monotone_score():
    """sqrt_softplus is increasing, so without bias and groups it selects the K
    largest logits; the weights are its scores, renormalised."""
    rng = np.random.default_rng(41)
    z = rng.standard_normal((20, 12)).astype(np.float32)
    r = O.route(z, 3, "sqrt_softplus", True)
    want = np.sort(np.argsort(-z, axis=1, kind="stable")[:, :3], axis=1)
    np.testing.assert_array_equal(r["topk_ids"], want)
    s = np.sqrt(np.log1p(np.exp(z.astype(np.float64))))
    w = np.take_along_axis(s, want, axis=1)
    np.testing.assert_allclose(r["topk_weights"], w / w.sum(1, keepdims=True), rtol=1e-6)


def test_permute_align_golden_case():
    vals = {}
    for line in _golden_lines("permute_align_case.txt"):
        key, *rest = line.split()
        vals[key] = [int(v) for v in rest]
    ids = np.array(vals["topk_ids"], dtype=np.int32).reshape(3, 2)
    r = O.permute_align(ids, 3, 4)
    assert int(r["num_tokens_post_pad"]) == vals["num_tokens_post_pad"][0]
    np.testing.assert_array_equal(r["sorted_token_ids"], vals["sorted_token_ids"])
    np.testing.assert_array_equal(r["expert_ids"], vals["expert_ids"])


@pytest.mark.parametrize("T,K,E,bs", [(37, 3, 5, 16), (1, 1, 1, 64), (50, 8, 64, 8), (9, 2, 40, 4)])
def test_permute_align_invariants(T, K, E, bs):
    """Each expert's range holds exactly its routes, then numel; the ranges
    follow in expert order, each a multiple of block_size long (empty experts
    take none); expert_ids names each block's owner; the rest is padding."""
    rng = np.random.default_rng(T * 100 + E)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    r = O.permute_align(ids, E, bs)
    flat = ids.reshape(-1)
    numel = flat.size
    sid, eid = r["sorted_token_ids"], r["expert_ids"]
    assert sid.size == numel + (E + 1) * (bs - 1) and eid.size == -(-sid.size // bs)
    pos = 0
    for e in range(E):
        routes = np.nonzero(flat == e)[0]
        padded = -(-len(routes) // bs) * bs
        blk = sid[pos:pos + padded]
        assert sorted(blk[:len(routes)].tolist()) == routes.tolist()
        assert (blk[len(routes):] == numel).all()
        assert (eid[pos // bs:(pos + padded) // bs] == e).all()
        pos += padded
    assert int(r["num_tokens_post_pad"]) == pos
    assert (sid[pos:] == numel).all() and ((eid[pos // bs:] < 0) | (eid[pos // bs:] >= E)).all()


def test_grouped_gemm_layouts_against_row_loops():
    """per_row and masked rows against explicit loops: out[row] = a[row] @
    b[expert of row]^T (+ bias, activation), every valid row, nothing else."""
    rng = np.random.default_rng(51)
    E, K, N = 4, 6, 5
    b = rng.standard_normal((E, N, K))
    bias = rng.standard_normal((E, N))
    ids = np.array([0, 0, 2, 2, 2, 3])              # expert 1 empty
    a = rng.standard_normal((ids.size, K))
    got = O.grouped_gemm_layout(a, b, "per_row", ids, bias=bias, dtype=None)
    for r, e in enumerate(ids):
        np.testing.assert_allclose(got[r], a[r] @ b[e].T + bias[e], rtol=1e-13)
    am = rng.standard_normal((E, 3, K))
    counts = [2, -1, 9, 0]                           # clamped to 2, 0, 3, 0
    got = O.grouped_gemm_layout(am, b, "masked", counts, act=O.ACT_RELU, F=N, dtype=None)
    for e, m in enumerate([2, 0, 3, 0]):
        for r in range(3):
            if r < m:
                np.testing.assert_allclose(got[e, r], np.maximum(am[e, r] @ b[e].T, 0), rtol=1e-13)
            else:
                assert np.isnan(got[e, r]).all()


def test_swiglu_fusion0_two_tensors_against_row_loops():
    """SwiGLU fusion 0 (gate from FC1, up from FC3, two tensors): every row
    against an explicit loop over its expert's two projections."""
    rng = np.random.default_rng(61)
    E, K, F = 3, 5, 4
    wg, wu = rng.standard_normal((E, F, K)), rng.standard_normal((E, F, K))
    bg, bu = rng.standard_normal((E, F)), rng.standard_normal((E, F))
    seg_end = np.array([2, 2, 5])
    a = rng.standard_normal((5, K)) * 3
    got = O.grouped_gemm_act_split(a, wg, wu, seg_end, O.ACT_SWIGLU, 2.0, 1.5, 0.5, bg, bu,
                                   dtype=None)
    for r in range(5):
        e = int(np.searchsorted(seg_end, r, side="right"))
        g = a[r] @ wg[e].T + bg[e]
        l = a[r] @ wu[e].T + bu[e]
        G, L = np.minimum(g, 2.0), np.clip(l, -2.0, 2.0)
        np.testing.assert_allclose(got[r], G / (1 + np.exp(-1.5 * G)) * (L + 0.5), rtol=1e-13)


def test_planted_mistakes_are_caught(monkeypatch):
    """A wrong sign in the sigmoid, swapped gate/up halves, or ties to the higher
    index each make one of the pins above fail."""
    orig = O.sigmoid64
    monkeypatch.setattr(O, "sigmoid64", lambda x: orig(-np.asarray(x)))
    with pytest.raises(AssertionError):
        test_swiglu_golden_points()
    monkeypatch.setattr(O, "sigmoid64", orig)

    # the shared expert: a flipped sigmoid, swapped gate/up halves or a
    # transposed down weight each fail its golden points
    monkeypatch.setattr(O, "sigmoid64", lambda x: orig(-np.asarray(x)))
    with pytest.raises(AssertionError):
        test_shared_expert_golden_points()
    monkeypatch.setattr(O, "sigmoid64", orig)
    orig_shared = O.shared_expert_mlp

    def swapped(hidden, w_gate_up, w_down, dtype="bf16"):
        S = np.asarray(w_gate_up).shape[0] // 2
        w = np.concatenate([np.asarray(w_gate_up)[S:], np.asarray(w_gate_up)[:S]])
        return orig_shared(hidden, w, w_down, dtype)

    for bad in (swapped, lambda h, gu, d, dtype="bf16": orig_shared(h, gu, np.asarray(d).T, dtype)):
        monkeypatch.setattr(O, "shared_expert_mlp", bad)
        with pytest.raises(AssertionError):
            test_shared_expert_golden_points()
    monkeypatch.setattr(O, "shared_expert_mlp", orig_shared)

    # fp8: a wrong exponent bias, or the b scale taken per row block instead
    # of per column block, each fail a pin
    orig_dec = O.e4m3_to_float
    monkeypatch.setattr(O, "e4m3_to_float", lambda c: orig_dec(c) * 2.0)
    with pytest.raises(AssertionError):
        test_e4m3_golden_points()
    monkeypatch.setattr(O, "e4m3_to_float", orig_dec)
    orig_fp8 = O.grouped_gemm_fp8_masked

    def scale_swapped(a, sa, b, sb, counts, dtype="bf16"):
        return orig_fp8(a, sa, b, np.ascontiguousarray(np.asarray(sb)[:, ::-1]), counts, dtype)

    monkeypatch.setattr(O, "grouped_gemm_fp8_masked", scale_swapped)
    with pytest.raises(AssertionError):
        test_fp8_scales_act_per_block()
    monkeypatch.setattr(O, "grouped_gemm_fp8_masked", orig_fp8)

    # expert parallelism: a rank that forgets weight_scale breaks the sum
    orig_local = O.ffn_forward_local
    monkeypatch.setattr(O, "ffn_forward_local",
                        lambda x, rp, ws, *a, **k: orig_local(x, rp, np.ones_like(ws), *a, **k))
    with pytest.raises(AssertionError):
        test_expert_parallel_slices_sum_to_the_layer()
    monkeypatch.setattr(O, "ffn_forward_local", orig_local)

    # the tanh form of GELU instead of the exact one fails the points
    monkeypatch.setattr(O, "gelu64", lambda x: 0.5 * np.asarray(x) * (1 + np.tanh(
        math.sqrt(2 / math.pi) * (np.asarray(x) + 0.044715 * np.asarray(x) ** 3))))
    with pytest.raises(AssertionError):
        test_activation_and_score_golden_points()
    monkeypatch.undo()

    orig_split = O.split_gate_up
    monkeypatch.setattr(O, "split_gate_up", lambda P, F, f: orig_split(P, F, f)[::-1])
    with pytest.raises(AssertionError):
        test_silu_and_mul_layout_and_values()
    monkeypatch.setattr(O, "split_gate_up", orig_split)

    monkeypatch.setattr(O, "topk_ascending",
                        lambda u, K: np.sort(np.argsort(-u[:, ::-1], axis=1, kind="stable")[:, :K] * -1
                                             + u.shape[1] - 1, axis=1).astype(np.int32))
    with pytest.raises(AssertionError):
        test_routing_golden_cases()
