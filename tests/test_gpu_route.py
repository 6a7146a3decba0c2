"""Router kernel against the oracle: ids bit-exact, weights within 1e-5
relative (the pages allow 1e-4), MoERouter outputs, hash routing, ties and
edge cases."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_gb300 import synth
from oracle import moe_oracle as O
from oracle import cases

from gpu_cases import make, np_

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_ffn_gb300 import build, moe as m

    build.build()
    return m


def _route_both(moe, cfg, inp, ref):
    p, _ = moe.config_params(cfg)
    w, ids, probs, ws = moe.moe_route(inp["logits"], p, inp["correction_bias"], inp["expert_ids"])
    torch.cuda.synchronize()
    r = O.route(ref["logits"], cfg.K, cfg.scoring, cfg.renormalize, cfg.G, cfg.TG, cfg.rsf,
                ref["correction_bias"], ref["expert_ids"], cfg.local_start, cfg.local_count,
                cfg.route_scale)
    return (np_(w), np_(ids), None if probs is None else np_(probs),
            None if ws is None else np_(ws)), r


def _check_route(moe, cfg):
    inp, ref = make(cfg.replace(H=64, F=64))  # routing does not depend on H, F
    (w, ids, probs, wsc), r = _route_both(moe, cfg, inp, ref)
    np.testing.assert_array_equal(ids, r["topk_ids"])
    np.testing.assert_allclose(w, r["topk_weights"], rtol=1e-5)
    if cfg.local_count:
        sent = r["router_probs"] == -1e30
        np.testing.assert_array_equal(probs == np.float32(-1e30), sent)
        np.testing.assert_allclose(probs[~sent], r["router_probs"][~sent], rtol=0, atol=1e-5)
        np.testing.assert_allclose(wsc, r["weight_scale"], rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("name", list(synth.CONFIGS))
def test_route_configs(moe, name):
    _check_route(moe, synth.CONFIGS[name])


@pytest.mark.parametrize("name,over", [
    ("qwen3_bf16", dict(scoring="sqrt_softplus")),                # MoERouter slice outputs too
    ("deepseek_v3_bf16", dict(scoring="sqrt_softplus", T=2048)),  # correction bias, 8 groups
    ("kimi_k2_decode_bf16", dict(scoring="sqrt_softplus", T=300)),
])
def test_route_sqrt_softplus(moe, name, over):
    _check_route(moe, synth.CONFIGS[name].replace(**over))


@pytest.mark.parametrize("hash_ids", [False, True])
def test_route_decode_hash(moe, hash_ids):
    cfg = synth.CONFIGS["kimi_k2_decode_bf16"].replace(hash_ids=hash_ids, H=128, F=256,
                                                       local_start=100, local_count=64)
    inp, ref = make(cfg)
    (w, ids, probs, wsc), r = _route_both(moe, cfg, inp, ref)
    np.testing.assert_array_equal(ids, r["topk_ids"])
    np.testing.assert_allclose(w, r["topk_weights"], rtol=1e-5)
    sent = r["router_probs"] == -1e30
    np.testing.assert_array_equal(probs == np.float32(-1e30), sent)
    np.testing.assert_allclose(probs[~sent], r["router_probs"][~sent], atol=1e-5)
    np.testing.assert_allclose(wsc, r["weight_scale"], rtol=1e-5, atol=1e-7)


def test_route_ties_and_edges(moe):
    dev = "cuda"
    # equal logits: ids 0..K-1, weights 1/K
    z = torch.zeros((5, 16), device=dev)
    w, ids, _, _ = moe.moe_route(z, moe.route_params(4, "softmax", True))
    assert (np_(ids) == np.arange(4)).all()
    np.testing.assert_allclose(np_(w), 0.25, rtol=1e-6)
    # K = E selects everything, in ascending order
    z = torch.randn((33, 12), device=dev)
    w, ids, _, _ = moe.moe_route(z, moe.route_params(12, "sigmoid", False))
    assert (np_(ids) == np.arange(12)).all()
    # E = 1, K = 1
    z = torch.randn((7, 1), device=dev)
    w, ids, _, _ = moe.moe_route(z, moe.route_params(1, "softmax", True, routed_scaling_factor=2.0))
    assert (np_(ids) == 0).all()
    np.testing.assert_allclose(np_(w), 2.0, rtol=1e-6)
    # E not a multiple of 32, groups, bias, T = 1
    for E, G, TG, K in ((96, 4, 2, 6), (40, 8, 3, 5), (1000, 8, 4, 8), (250, 1, 1, 7)):
        cfg = synth.MoEConfig("edge", 9, T=1 if E == 250 else 77, H=8, F=8, E=E, K=K,
                              scoring="sigmoid", G=G, TG=TG, rsf=1.5, cbias_std=0.1 if G > 1 else None)
        inp, ref = make(cfg)
        (w, ids, _, _), r = _route_both(moe, cfg, inp, ref)
        np.testing.assert_array_equal(ids, r["topk_ids"])
        np.testing.assert_allclose(w, r["topk_weights"], rtol=1e-5)


@pytest.mark.parametrize("E,K,G,TG,scoring", [
    (1024, 64, 32, 32, "sigmoid"),   # the largest E, K and G accepted
    (1024, 64, 32, 8, "sigmoid"),    # group pruning at the largest G
    (1024, 8, 1, 1, "softmax"),
    (64, 64, 1, 1, "softmax"),       # K = E = 64
])
def test_route_maximum_sizes(moe, E, K, G, TG, scoring):
    cfg = synth.MoEConfig("max", 11, T=300, H=8, F=8, E=E, K=K, scoring=scoring, G=G, TG=TG,
                          rsf=2.5, cbias_std=0.1 if scoring == "sigmoid" else None,
                          local_start=max(0, E - 96), local_count=min(96, E))
    inp, ref = make(cfg)
    (w, ids, probs, wsc), r = _route_both(moe, cfg, inp, ref)
    np.testing.assert_array_equal(ids, r["topk_ids"])
    np.testing.assert_allclose(w, r["topk_weights"], rtol=1e-5)
    sent = r["router_probs"] == -1e30
    np.testing.assert_array_equal(probs == np.float32(-1e30), sent)
    np.testing.assert_allclose(probs[~sent], r["router_probs"][~sent], rtol=0, atol=1e-5)
    np.testing.assert_allclose(wsc, r["weight_scale"], rtol=1e-5, atol=1e-7)


def test_route_rejects_past_the_limits(moe):
    z = torch.randn((4, 1025), device="cuda")
    with pytest.raises(moe.MoEError):
        moe.moe_route(z, moe.route_params(8, "softmax", True))          # E > 1024
    z = torch.randn((4, 128), device="cuda")
    with pytest.raises(moe.MoEError):
        moe.moe_route(z, moe.route_params(65, "softmax", True))         # K > 64
    with pytest.raises(moe.MoEError):
        moe.moe_route(z, moe.route_params(8, "sigmoid", True, num_expert_group=64,
                                          topk_group=4))                # G > 32


def test_route_golden_cases_on_gpu(moe):
    import json
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "routing_cases.txt")
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c = json.loads(line)
        p = moe.route_params(c["K"], c["scoring"], c["renormalize"], c["G"], c["TG"], c["rsf"],
                             c.get("local_start", 0), c.get("local_count", 0),
                             c.get("route_scale", 1.0))
        z = torch.tensor(c["logits"], dtype=torch.float32, device="cuda")
        b = None if c["bias"] is None else torch.tensor(c["bias"], dtype=torch.float32, device="cuda")
        w, ids, probs, wsc = moe.moe_route(z, p, b)
        np.testing.assert_array_equal(np_(ids), np.array(c["ids"]), err_msg=c["name"])
        np.testing.assert_allclose(np_(w), np.array(c["weights"]), rtol=1e-6, err_msg=c["name"])
        if "router_probs" in c:
            np.testing.assert_allclose(np_(probs), np.array(c["router_probs"]), rtol=1e-6)
            np.testing.assert_allclose(np_(wsc), np.array(c["weight_scale"]), rtol=1e-6)


def _fused_vs_separate(moe, cfg, inp):
    p, _ = moe.config_params(cfg)
    w, ids, probs, wsc, maps = moe.moe_route_permute(inp["logits"], p, inp["correction_bias"],
                                                     inp["expert_ids"])
    w2, ids2, probs2, wsc2 = moe.moe_route(inp["logits"], p, inp["correction_bias"],
                                           inp["expert_ids"])
    perm = moe.moe_permute(ids2, cfg.E)
    torch.cuda.synchronize()
    assert moe.moe_sync_status(maps["ws"]) == moe.MOE_OK
    assert torch.equal(w, w2) and torch.equal(ids, ids2)
    if probs is not None:
        assert torch.equal(probs, probs2) and torch.equal(wsc, wsc2)
    for k in ("seg_end", "row_to_route", "route_to_row"):
        assert torch.equal(maps[k], perm[k]), k
    return ids


@pytest.mark.parametrize("name,T", [
    ("tiny_fp32", 64), ("qwen3_bf16", 4096), ("deepseek_v3_bf16", 8192),
    ("gpt_oss_bf16", 2048), ("kimi_k2_decode_bf16", 16),
    ("qwen3_bf16", 1), ("qwen3_bf16", 20000),   # one token; 157 chunks on 152 SMs
])
def test_route_permute_fused_matches_separate(moe, name, T):
    """The one-launch route + index maps equals moe_route then moe_permute bit
    for bit (ids, weights, MoERouter outputs, seg_end and both maps), and its
    maps equal the oracle's permutation of the oracle's routing."""
    cfg = synth.CONFIGS[name].replace(T=T, H=64, F=64)
    inp, ref = make(cfg)
    ids = _fused_vs_separate(moe, cfg, inp)
    r = O.route(ref["logits"], cfg.K, cfg.scoring, cfg.renormalize, cfg.G, cfg.TG, cfg.rsf,
                ref["correction_bias"], ref["expert_ids"], cfg.local_start, cfg.local_count,
                cfg.route_scale)
    np.testing.assert_array_equal(np_(ids), r["topk_ids"])


@pytest.mark.parametrize("E", [8, 384, 512])
def test_route_permute_fused_expert_counts(moe, E):
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=777, E=E, K=min(8, E), H=64, F=64,
                                              local_count=0)
    inp, _ = make(cfg)
    _fused_vs_separate(moe, cfg, inp)


def test_route_permute_fused_hash_and_bad_ids(moe):
    cfg = synth.CONFIGS["kimi_k2_decode_bf16"].replace(hash_ids=True, T=40, H=128, F=256)
    inp, _ = make(cfg)
    _fused_vs_separate(moe, cfg, inp)
    p, _ = moe.config_params(cfg)
    bad = inp["expert_ids"].clone()
    bad[3, 2] = cfg.E + 5
    *_, maps = moe.moe_route_permute(inp["logits"], p, inp["correction_bias"], bad)
    assert moe.moe_sync_status(maps["ws"]) == moe.MOE_ERR_DEVICE
    assert int(maps["seg_end"][-1]) == cfg.T * cfg.K - 1  # the bad route got no row


def test_route_permute_reuses_workspace(moe):
    """The grid-barrier counters reset themselves: launches back to back on one
    workspace (no status clear between them) give the same maps, and leave
    the counters (status bytes 16..27) at zero."""
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=3000, H=64, F=64)
    inp, _ = make(cfg)
    p, _ = moe.config_params(cfg)
    first = moe.moe_route_permute(inp["logits"], p, inp["correction_bias"])
    ws = first[4]["ws"]
    for _ in range(3):
        again = moe.moe_route_permute(inp["logits"], p, inp["correction_bias"], ws=ws)
        for k in ("seg_end", "row_to_route", "route_to_row"):
            assert torch.equal(again[4][k], first[4][k]), k
        assert torch.equal(again[1], first[1])
    assert moe.moe_sync_status(ws) == moe.MOE_OK
    assert int(ws[16:28].count_nonzero()) == 0


@pytest.mark.parametrize("dtype,H", [("bf16", 2048), ("bf16", 100), ("f32", 64)])
def test_permute_gather_after_fused_maps(moe, dtype, H):
    """The gather step on its own, from the maps of the one-launch route +
    permute, equals moe_permute's permuted copy bit for bit (16-byte rows and
    ragged rows)."""
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=777, H=H, F=64, local_count=0)
    inp, _ = make(cfg)
    p, _ = moe.config_params(cfg)
    hidden = inp["hidden"].to(synth.torch_dtype(dtype))
    _, ti, _, _, maps = moe.moe_route_permute(inp["logits"], p, inp["correction_bias"])
    got = moe.moe_permute_gather(hidden, maps["seg_end"], maps["row_to_route"], cfg.K)
    ref = moe.moe_permute(ti, cfg.E, hidden)
    torch.cuda.synchronize()
    assert torch.equal(got, ref["expert_input"])


def test_route_permute_rejects_large_e(moe):
    cfg = synth.CONFIGS["qwen3_bf16"].replace(T=8, E=640, K=8, H=64, F=64, local_count=0)
    inp, _ = make(cfg)
    p, _ = moe.config_params(cfg)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_route_permute(inp["logits"], p)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
