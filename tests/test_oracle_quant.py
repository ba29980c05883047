"""Pins of the oracle's group-32 quantize / dequantize (page
"code/flashsim/quantization.py", Algorithms 2-3) against things other than the
oracle itself: hand-worked groups, numpy's float16 rounding, brute-force
nearest-code search in binary64, symmetries, and error bounds.
"""

import json
import os

import numpy as np
import pytest

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantize_single_groups.json")


def _group(case):
    x = np.zeros(32, np.float32)
    if "x" in case:
        x[: len(case["x"])] = case["x"]
    else:
        x[:] = case["x_fill"]
    return x


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_worked_groups(case):
    x = _group(case)
    codes, scales = O.quantize(x, case["spec"])
    assert scales.shape == (1,)
    assert scales[0] == int(case["scale_f16_bits"], 16)
    sv = O.f16_bits_to_f32(scales)[0]
    exp_sv = float(case["scale_value"])
    assert (np.isinf(sv) and np.isinf(exp_sv)) or sv == np.float32(exp_sv)
    if "codes" in case:
        k = len(case["codes"])
        assert codes[:k].astype(int).tolist() == case["codes"]
        assert np.all(codes[k:] == 0)
    else:
        assert np.all(codes.astype(int) == case["codes_fill"])
    if "dequant" in case:
        d = O.dequantize(codes, scales, case["spec"])
        k = len(case["dequant"])
        exp = np.array([float(v) for v in case["dequant"]])
        got = d[:k].astype(np.float64)
        nan = np.isnan(exp)
        assert np.array_equal(np.isnan(got), nan)
        np.testing.assert_allclose(got[~nan], exp[~nan], rtol=2e-7, atol=0)


def test_zero_scale_gives_zero_codes():
    x = W.battery()["tiny"].numpy()
    for spec in ("momentum", "variance"):
        xin = np.abs(x) if spec == "variance" else x
        codes, scales = O.quantize(xin, spec)
        assert np.all(scales == 0)
        assert np.all(codes == 0)
        assert np.all(O.dequantize(codes, scales, spec) == 0)


def test_code_ranges_on_battery():
    for name, t in W.battery().items():
        x = t.numpy()
        c, _ = O.quantize(x, "momentum")
        assert c.min() >= -127 and c.max() <= 127, name
        c, _ = O.quantize(np.abs(x), "variance")
        assert c.dtype == np.uint8


@pytest.mark.parametrize("spec", ["momentum", "variance", "momentum_linear", "variance_linear"])
def test_ragged_tail_is_zero_padded(spec):
    x = W.battery()["nonmult32"].numpy()
    if spec.startswith("variance"):
        x = np.abs(x)
    n = x.size
    assert n % 32 == 17
    padded = np.concatenate([x, np.zeros(32 - n % 32, np.float32)])
    c1, s1 = O.quantize(x, spec)
    c2, s2 = O.quantize(padded, spec)
    assert s1.size == (n + 31) // 32
    assert np.array_equal(c1, c2[:n]) and np.array_equal(s1, s2)
    # padding is 0 and every group max is >= 0, so the tail group's scale is the
    # fp16 of the max over its 17 live elements
    tail = x[-17:]
    ref = np.float16(np.sqrt(tail).max() if spec == "variance" else
                     (np.abs(tail).max() if spec.startswith("momentum") else tail.max()))
    assert s1[-1] == ref.view(np.uint16)


@pytest.mark.parametrize("spec", ["momentum", "variance"])
def test_scales_are_numpy_float16_of_group_max(spec):
    x = W.battery()["heavy_tail"].numpy()[: 1 << 16]
    x = np.abs(x) if spec == "variance" else x
    _, s = O.quantize(x, spec)
    g = x.reshape(-1, 32).astype(np.float32)
    gm = np.sqrt(g).max(axis=1) if spec == "variance" else np.abs(g).max(axis=1)
    with np.errstate(over="ignore"):
        ref = gm.astype(np.float16).view(np.uint16)
    assert np.array_equal(s, ref)


def test_momentum_odd_symmetry():
    x = W.battery()["normal"].numpy()
    c1, s1 = O.quantize(x, "momentum")
    c2, s2 = O.quantize(-x, "momentum")
    assert np.array_equal(s1, s2)
    assert np.array_equal(c2.astype(int), -c1.astype(int))


@pytest.mark.parametrize("k", [-3, 2, 5])
def test_power_of_two_invariance(k):
    x = W.battery()["normal"].numpy()
    cm, sm = O.quantize(x, "momentum")
    cm2, sm2 = O.quantize(x * np.float32(2.0 ** k), "momentum")
    sv, sv2 = O.f16_bits_to_f32(sm), O.f16_bits_to_f32(sm2)
    # only groups whose scale is a normal fp16 number before and after
    ok = (sv >= 2 ** -14) & (sv * 2.0 ** k >= 2 ** -14) & (sv * 2.0 ** k < 65504)
    assert ok.mean() > 0.99
    np.testing.assert_array_equal(sv2[ok], (sv[ok] * 2.0 ** k).astype(np.float32))
    rows = np.repeat(ok, 32)
    np.testing.assert_array_equal(cm2[rows], cm[rows])
    xv = np.abs(x)
    cv, svb = O.quantize(xv, "variance")
    cv2, svb2 = O.quantize(xv * np.float32(4.0 ** k), "variance")
    a, b = O.f16_bits_to_f32(svb), O.f16_bits_to_f32(svb2)
    ok = (a >= 2 ** -14) & (a * 2.0 ** k >= 2 ** -14) & (a * 2.0 ** k < 65504)
    np.testing.assert_array_equal(b[ok], (a[ok] * 2.0 ** k).astype(np.float32))
    np.testing.assert_array_equal(cv2[np.repeat(ok, 32)], cv[np.repeat(ok, 32)])


@pytest.mark.parametrize("spec", ["momentum", "variance", "momentum_linear", "variance_linear"])
def test_brute_force_nearest_code(spec):
    """The chosen code is the nearest of all codes to the companded value, which
    is evaluated in binary64 from the stored fp16 scale (numpy float16)."""
    rng = np.random.default_rng(17)
    x = (rng.standard_normal(4096) * np.exp(rng.standard_normal(4096))).astype(np.float32)
    signed = spec.startswith("momentum")
    if not signed:
        x = np.abs(x)
    codes, scales = O.quantize(x, spec)
    g = x.reshape(-1, 32).astype(np.float64)
    if spec == "variance":
        g = np.sqrt(g)
    amax = (np.abs(g) if signed else g).max(axis=1, keepdims=True)
    s = amax.astype(np.float16).astype(np.float64)
    assert np.array_equal(s.reshape(-1).astype(np.float16).view(np.uint16), scales)
    y = g / np.where(s == 0, 1.0, s)
    if spec == "momentum":
        y = 2 * y / (1 + np.abs(y))
    qmax = 127 if signed else 255
    cand = np.arange(-127, 128) if signed else np.arange(0, 256)
    dist = np.abs(y.reshape(-1, 1) * qmax - cand.reshape(1, -1))
    best = dist.min(axis=1)
    mine = np.abs(y.reshape(-1) * qmax - codes.astype(np.float64))
    # ties and binary32-vs-binary64 rounding leave a sliver of slack
    assert np.all(mine <= best + 1e-4)


def test_group_max_maps_to_top_code():
    x = W.battery()["normal"].numpy()
    c, s = O.quantize(x, "momentum")
    g = x.reshape(-1, 32)
    arg = np.abs(g).argmax(axis=1)
    top = c.reshape(-1, 32)[np.arange(g.shape[0]), arg].astype(int)
    assert np.all(np.abs(top) == 127)
    cv, _ = O.quantize(np.abs(x), "variance")
    topv = cv.reshape(-1, 32)[np.arange(g.shape[0]), arg]
    assert np.all(topv == 255)


def test_codes_monotone_within_group():
    x = W.battery()["normal"].numpy()
    for spec, xin in (("momentum", x), ("variance", np.abs(x))):
        c, _ = O.quantize(xin, spec)
        g = xin.reshape(-1, 32)
        order = np.argsort(g, axis=1, kind="stable")
        cs = np.take_along_axis(c.reshape(-1, 32).astype(int), order, axis=1)
        assert np.all(np.diff(cs, axis=1) >= 0), spec


def test_roundtrip_error_bounds():
    """Half a code step in the companded domain, pulled back through the inverse
    companding (slope <= 2 for softsign on [-1, 1]; sqrt domain for variance),
    plus the clamp excess max(0, |x| - s) where the fp16 scale rounded below
    the group max (coarse subnormal scales)."""
    for name in ("normal", "heavy_tail", "nonmult32", "with_zeros", "adam_v_like"):
        x = W.battery()[name].numpy()
        n = x.size
        c, s = O.quantize(x, "momentum")
        d = O.dequantize(c, s, "momentum").astype(np.float64)
        sv = np.repeat(O.f16_bits_to_f32(s).astype(np.float64), 32)[:n]
        fin = np.isfinite(sv)
        err = np.abs(d - x)[fin]
        excess = np.maximum(0.0, np.abs(x.astype(np.float64)) - sv)[fin]
        assert np.all(err <= sv[fin] * (1.0 / 127) * (1 + 1e-3) + excess * (1 + 1e-6) + 1e-30), name
        xv = np.abs(x)
        cv, svb = O.quantize(xv, "variance")
        dv = O.dequantize(cv, svb, "variance").astype(np.float64)
        sv = np.repeat(O.f16_bits_to_f32(svb).astype(np.float64), 32)[:n]
        fin = np.isfinite(sv)
        r = np.sqrt(xv.astype(np.float64))
        err = np.abs(np.sqrt(dv) - r)[fin]
        excess = np.maximum(0.0, r - sv)[fin]
        assert np.all(err <= sv[fin] * (0.5 / 255) * (1 + 1e-3) + excess * (1 + 1e-6) + 1e-30), name


def test_overflow_groups_in_heavy_tail():
    """fp16 scale overflow is followed literally: codes 0, dequantized NaN."""
    x = W.battery()["heavy_tail"].numpy()
    c, s = O.quantize(x, "momentum")
    inf_groups = s == 0x7C00
    assert inf_groups.sum() > 0
    assert np.all(c.reshape(-1, 32)[inf_groups] == 0)
    d = O.dequantize(c, s, "momentum").reshape(-1, 32)
    assert np.all(np.isnan(d[inf_groups]))
    assert np.all(np.isfinite(d[~inf_groups]))


def test_nmse_report_is_sane():
    """No expected NMSE values are printed on the pages; these are loose sanity
    gates only (a broken code path gives NMSE of order 1)."""
    out = {}
    for name, t in W.battery().items():
        x = t.numpy()
        c, s = O.quantize(x, "momentum")
        out[name, "m"] = O.nmse(x, O.dequantize(c, s, "momentum"))
        xv = np.abs(x)
        c, s = O.quantize(xv, "variance")
        out[name, "v"] = O.nmse(xv, O.dequantize(c, s, "variance"))
    assert out["normal", "m"] < 1e-3 and out["normal", "v"] < 1e-3
    assert out["tiny", "m"] == pytest.approx(1.0) and out["tiny", "v"] == pytest.approx(1.0)
    assert out["const_groups", "m"] < 1e-6
    assert O.nmse(np.zeros(4), np.ones(4)) == 0.0
