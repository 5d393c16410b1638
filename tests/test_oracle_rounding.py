"""Pins for the oracle's rounding to the I/O formats.

The oracle rounds float64 results onto the fp32 / bf16 / fp16 grids with its
own routine. It is pinned here against things that do not share its formula:
exhaustive nearest-value search over every finite bf16 and fp16 bit pattern,
numpy's own float64 -> float32 / float16 casts, and torch's float32 -> bf16 cast.
"""

import numpy as np
import pytest
import torch

from oracle import round_to_format


def _all_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32).astype(np.float64)
    return bits.astype(np.uint16), vals


def _all_f16():
    bits = np.arange(1 << 16, dtype=np.uint16)
    return bits, bits.view(np.float16).astype(np.float64)


def _brute_nearest(v, bits, vals):
    """Nearest finite grid value by exhaustive search, ties to the even pattern.

    Values beyond the largest finite number by half a spacing or more go to inf.
    """
    finite = np.isfinite(vals)
    fb, fv = bits[finite], vals[finite]
    order = np.argsort(fv, kind="stable")
    fb, fv = fb[order], fv[order]
    # drop -0 duplicates so each value appears once (keep +0)
    keep = ~((fv == 0) & (np.signbit(fv)))
    fb, fv = fb[keep], fv[keep]
    out = np.empty_like(v)
    vmax = fv[-1]
    spacing_top = fv[-1] - fv[-2]
    for i, x in enumerate(v):
        if abs(x) >= vmax + spacing_top / 2:
            out[i] = np.copysign(np.inf, x)
            continue
        d = np.abs(fv - x)
        m = d.min()
        cand = np.nonzero(d == m)[0]
        if len(cand) == 1:
            out[i] = fv[cand[0]]
        else:
            even = [c for c in cand if (int(fb[c]) & 1) == 0]
            assert len(even) == 1
            out[i] = fv[even[0]]
        if out[i] == 0:
            out[i] = np.copysign(0.0, x)
    return out


def _probe_values(vals, rng, n_random):
    """Random doubles plus exact midpoints and near-midpoints of the grid."""
    fv = np.unique(vals[np.isfinite(vals)])
    idx = rng.integers(0, len(fv) - 1, size=n_random)
    lo, hi = fv[idx], fv[idx + 1]
    mid = (lo + hi) / 2
    t = rng.random(n_random)
    inside = lo + t * (hi - lo)
    nudged = np.nextafter(mid, np.where(rng.random(n_random) < 0.5, -np.inf, np.inf))
    return np.concatenate([mid, inside, nudged, [0.0, -0.0, fv[0], fv[-1]]])


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_round_matches_exhaustive_nearest(fmt):
    rng = np.random.default_rng(1)
    bits, vals = _all_bf16() if fmt == "bf16" else _all_f16()
    v = _probe_values(vals, rng, 700)
    got = round_to_format(v, fmt)
    want = _brute_nearest(v, bits, vals)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(np.signbit(got), np.signbit(want))


def test_round_f32_matches_numpy_cast():
    rng = np.random.default_rng(2)
    v = np.concatenate([
        rng.standard_normal(20000) * np.exp2(rng.integers(-140, 128, 20000)),
        np.ldexp(rng.random(2000), -149),             # fp32 subnormal range
        [np.ldexp(1.0 + 2.0 ** -24, 0), np.ldexp(1.0 + 3 * 2.0 ** -24, 0),  # ties
         3.4028235677973366e38, 3.4028235e38 * 1.0000001, np.inf, -np.inf, 0.0, -0.0],
    ])
    with np.errstate(over="ignore"):
        want = v.astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(round_to_format(v, "f32"), want)


def test_round_f16_matches_numpy_cast():
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.standard_normal(20000) * np.exp2(rng.integers(-26, 17, 20000)),
        [65504.0, 65519.99, 65520.0, 2.0 ** -25, 2.0 ** -25 * 1.0001, 3 * 2.0 ** -25],
    ])
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(round_to_format(v, "f16"), want)


def test_round_bf16_matches_torch_cast_of_fp32_values():
    # torch rounds float32 -> bfloat16 to nearest-even; feeding values that
    # are exact in float32 makes that a single rounding, like the oracle's.
    rng = np.random.default_rng(4)
    v32 = (rng.standard_normal(50000) * np.exp2(rng.integers(-130, 120, 50000))).astype(np.float32)
    want = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(round_to_format(v32.astype(np.float64), "bf16"), want)


def test_round_f64_is_identity_and_keeps_nan():
    v = np.array([1.0 + 2.0 ** -52, np.nan, -np.inf])
    out = round_to_format(v, "f64")
    assert out[0] == v[0] and np.isnan(out[1]) and out[2] == -np.inf
    assert np.isnan(round_to_format(np.array([np.nan]), "bf16")[0])


def _all_e4m3():
    """Every E4M3 code decoded by hand from its bit fields (NaN codes dropped)."""
    vals, codes = [], []
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            continue                      # NaN
        if e == 0:
            v = sign * m * 2.0 ** -9      # subnormal
        else:
            v = sign * (1 + m / 8.0) * 2.0 ** (e - 7)
        vals.append(v)
        codes.append(c)
    return np.array(codes), np.array(vals)


def test_e4m3_matches_exhaustive_nearest_with_saturation():
    from oracle import round_to_e4m3_satfinite
    codes, vals = _all_e4m3()
    assert vals.max() == 448.0 and vals.min() == -448.0
    rng = np.random.default_rng(5)
    fv = np.unique(vals)
    idx = rng.integers(0, len(fv) - 1, size=3000)
    lo, hi = fv[idx], fv[idx + 1]
    probe = np.concatenate([(lo + hi) / 2, lo + rng.random(3000) * (hi - lo),
                            [0.0, -0.0, 448.0, 449.0, 464.0, 470.0, 1e6, -1e6, 2.0 ** -10,
                             3 * 2.0 ** -10, -2.0 ** -11]])
    got = round_to_e4m3_satfinite(probe)
    for x, g in zip(probe, got):
        if abs(x) >= 448.0:
            assert g == np.copysign(448.0, x)
            continue
        d = np.abs(fv - x)
        cand = np.nonzero(d == d.min())[0]
        if len(cand) == 1:
            want = fv[cand[0]]
        else:                              # tie: the code with an even mantissa
            even = [fv[i] for i in cand
                    if int(codes[vals == fv[i]][0]) & 1 == 0]
            assert len(even) == 1
            want = even[0]
        assert g == want or (g == 0 and want == 0), (x, g, want)
    assert np.isnan(round_to_e4m3_satfinite(np.array([np.nan]))[0])


def test_e4m3_matches_torch_cast_in_range():
    from oracle import round_to_e4m3_satfinite
    rng = np.random.default_rng(6)
    v32 = (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 8, 20000))).astype(np.float32)
    v32 = v32[np.abs(v32) < 440.0]
    want = torch.from_numpy(v32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(round_to_e4m3_satfinite(v32.astype(np.float64)), want)


def test_fp8_quantize_multiplies_in_fp32():
    from oracle import quantize_fp8_e4m3
    y = np.array([1.0, -0.3125, 3.0, 1e3])
    out = quantize_fp8_e4m3(y, 2.0)
    np.testing.assert_array_equal(out, [2.0, -0.625, 6.0, 448.0])
