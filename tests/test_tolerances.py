"""Host checks of the parity helpers in tolerances.py: the secondary bound
admits exactly the roundings it is derived from (one flip of each route
output, half an ulp of the output's cast) and rejects an error one flip
larger; the stated bound is the plain 2e-2 * RMS(ref)."""
import numpy as np
import pytest

from tolerances import assert_forward_close, assert_layer_close, figures, flip_budget, ulp_bf16


def _case(seed=0, T=64, K=4, H=32):
    g = np.random.default_rng(seed)
    w = g.random((T, K))
    w /= w.sum(1, keepdims=True)
    y = g.standard_normal((T * K, H))
    y = y.astype(np.float32).astype(np.float64)
    exact = np.einsum("tk,tkh->th", w, y.reshape(T, K, H))
    return {"out_unrounded": exact, "route_out": y, "topk_weights": w}


def test_flip_budget_is_the_weighted_ulps():
    o = _case()
    b = flip_budget(o["route_out"], o["topk_weights"], "bf16")
    T, K = o["topk_weights"].shape
    want = sum(o["topk_weights"][:, k:k + 1] * ulp_bf16(o["route_out"][k::K]) for k in range(K))
    np.testing.assert_allclose(b, want, rtol=1e-12)


def test_secondary_admits_one_flip_per_route_and_the_final_cast():
    o = _case(1)
    T, K = o["topk_weights"].shape
    # every route output one ulp off in the worst direction, then the cast
    y2 = o["route_out"] + ulp_bf16(o["route_out"]) * np.sign(o["out_unrounded"]).repeat(K, 0)
    got = np.einsum("tk,tkh->th", o["topk_weights"], y2.reshape(T, K, -1))
    got = got + 0.5 * ulp_bf16(got) * np.sign(got)
    r = assert_forward_close(got, o, "bf16", "planted flips", stated=False)
    assert r["n_above_secondary"] == 0


def test_secondary_rejects_an_error_past_its_budget():
    o = _case(2)
    got = o["out_unrounded"].copy()
    rms = float(np.sqrt(np.mean(got ** 2)))
    lim = 2e-2 * rms + 0.5 * ulp_bf16(got[3, 5]) + flip_budget(
        o["route_out"], o["topk_weights"], "bf16")[3, 5]
    got[3, 5] += 1.01 * lim + ulp_bf16(got[3, 5])
    with pytest.raises(AssertionError):
        assert_forward_close(got, o, "bf16", "planted error", stated=False)


def test_stated_bound_is_two_percent_of_rms():
    exact = np.linspace(-1, 1, 1001)
    rms = float(np.sqrt(np.mean(exact ** 2)))
    got = exact.copy()
    got[10] += 0.019 * rms
    assert figures(got, exact, "bf16")["n_above_stated"] == 0
    assert_layer_close(got, exact, "bf16", "inside")
    got[10] += 0.002 * rms
    assert figures(got, exact, "bf16")["n_above_stated"] == 1
    with pytest.raises(AssertionError):
        assert_layer_close(got, exact, "bf16", "outside")
