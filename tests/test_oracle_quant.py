"""Pins for the oracle's quantisation and dequantisation.

[CG §2.3(1)] torch_quant_vectorized: MAX = bins // 2 - 1, max1 = amax |x|,
xq = round(x * MAX / max1 + MAX). [CG §2.4(2)] do_dequantize:
(t - MAX) / MAX * max1. The checks below come from the mathematics, not from
the oracle's own code: exact rational values, closed-form special cases,
constructed ties, monotonicity and the error bound.
"""
from fractions import Fraction

import numpy as np
import pytest

pytestmark = []


def _finite_halves():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    return h[np.isfinite(h)]


def _round_half_even(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def test_finite_half_count():
    assert _finite_halves().size == 63488


@pytest.mark.parametrize("bins", [4, 5, 8, 16, 32, 255, 256])
def test_closed_form_special_values(oracle_mod, bins):
    MAX = bins // 2 - 1
    for m in [1.0, 0.0999755859375, 18.78125, 65504.0, 6.103515625e-05]:
        x = np.array([m, -m, 0.0, m], np.float16)
        q, max1 = oracle_mod.quantize_group(x, bins)
        assert np.float16(m).view(np.uint16) == max1
        assert list(q) == [2 * MAX, 0, MAX, 2 * MAX]
        # dequantisation hits +-max1 and 0 exactly
        assert oracle_mod.dequantize_value(2 * MAX, bins, max1) == float(np.float16(m))
        assert oracle_mod.dequantize_value(0, bins, max1) == -float(np.float16(m))
        assert oracle_mod.dequantize_value(MAX, bins, max1) == 0.0


def test_all_zero_group_maps_to_offset(oracle_mod):
    for bins in (4, 16, 32, 256):
        x = np.array([0.0, -0.0, 0.0], np.float16)
        q, max1 = oracle_mod.quantize_group(x, bins)
        assert max1 == 0
        assert (q == bins // 2 - 1).all()
        assert oracle_mod.dequantize_value(int(q[0]), bins, max1) == 0.0


def test_ties_round_to_even(oracle_mod):
    # max1 = 1.875, bins = 32: MAX = 15 and factor = 15 / 1.875 = 8 exactly, so
    # x * factor + MAX lands exactly on .5 for these x; torch.round rounds
    # half to even (half-away-from-zero would give 16, 17, 15, 14).
    x = np.array([1.875, 0.0625, 0.1875, -0.0625, -0.1875], np.float16)
    q, _ = oracle_mod.quantize_group(x, 32)
    assert list(q[1:]) == [16, 16, 14, 14]


def test_nonfinite_rejected(oracle_mod):
    for bad in (np.inf, -np.inf, np.nan):
        x = np.array([1.0, bad], np.float16)
        with pytest.raises(oracle_mod.OracleError) as e:
            oracle_mod.quantize_group(x, 16)
        assert e.value.code == oracle_mod.ERR_NONFINITE


@pytest.mark.parametrize("bins", [3, 257, 0, -4])
def test_bad_bins_rejected(oracle_mod, bins):
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.quantize_group(np.ones(4, np.float16), bins)


@pytest.mark.parametrize("bins", [4, 8, 16, 32, 33, 256])
@pytest.mark.parametrize("max1", [1.0, 1.875, 0.0999755859375, 18.78125, 3.0517578125e-05, 60000.0])
def test_every_fp16_against_exact_rational(oracle_mod, bins, max1):
    """All finite fp16 x with |x| <= max1, each in the group [max1, x]: q is in
    [0, 2*MAX], monotone in x, and equals the exactly rounded value of the real
    x*MAX/max1 + MAX except within binary32 rounding of a .5 tie."""
    MAX = bins // 2 - 1
    h = _finite_halves()
    m16 = np.float16(max1)
    xs = np.sort(h[np.abs(h.astype(np.float64)) <= float(m16)].astype(np.float64)).astype(np.float16)
    groups = np.stack([np.full(xs.size, m16), xs], axis=1)  # [N, 2]
    k = groups[None]  # L=1, T=N, C=2
    sym, mx = oracle_mod.quantize(k, k, [bins], [bins])
    q = sym[0, 0, :, 1].astype(np.int64)
    assert (mx[0, 0] == m16.view(np.uint16)).all()
    assert q.min() >= 0 and q.max() <= 2 * MAX
    assert (np.diff(q) >= 0).all(), "q must be monotone in x"
    # exact real value, in float64 (x*MAX exact; one rounding in the division)
    y = xs.astype(np.float64) * MAX / float(m16) + MAX
    frac = y - np.floor(y)
    clear = np.abs(frac - 0.5) > 2.0 ** -14
    assert (q[clear] == np.floor(y[clear] + 0.5)).all()
    # near ties: one of the two neighbours; where MAX/max1 and x*MAX/max1 are
    # exact binary32 values the arithmetic is exact and a tie rounds to even
    exact_factor = Fraction(MAX) / Fraction(float(m16))
    factor_is_exact = Fraction(float(np.float32(exact_factor))) == exact_factor
    for i in np.nonzero(~clear)[0]:
        fr = Fraction(float(xs[i])) * MAX / Fraction(float(m16)) + MAX
        lo = fr.numerator // fr.denominator
        assert q[i] in (lo, lo + 1)
        prod = Fraction(float(xs[i])) * exact_factor
        if (fr - lo == Fraction(1, 2) and factor_is_exact
                and Fraction(float(np.float32(prod))) == prod):
            assert q[i] == _round_half_even(fr)


@pytest.mark.parametrize("bins", [4, 8, 16, 32, 256])
def test_error_bound_every_fp16(oracle_mod, bins):
    """|x - x^| <= max1 / (2 MAX) + one fp16 ulp of max1, for every finite x."""
    MAX = bins // 2 - 1
    h = _finite_halves()
    for max1 in (np.float16(1.0), np.float16(0.0999755859375), np.float16(512.0)):
        xs = h[np.abs(h.astype(np.float64)) <= float(max1)]
        groups = np.stack([np.full(xs.size, max1), xs], axis=1)[None]
        sym, mx = oracle_mod.quantize(groups, groups, [bins], [bins])
        xk, _ = oracle_mod.dequantize(sym, mx, [bins], [bins])
        err = np.abs(xk[0, :, 1].astype(np.float64) - xs.astype(np.float64))
        ulp = float(np.spacing(max1))
        assert err.max() <= float(max1) / (2 * MAX) + ulp


def test_dequantize_antisymmetric(oracle_mod):
    for bins in (4, 16, 32, 256):
        MAX = bins // 2 - 1
        for m in (1.0, 0.3, 1000.0):
            mb = int(np.float16(m).view(np.uint16))
            for q in range(0, 2 * MAX + 1):
                a = oracle_mod.dequantize_value(q, bins, mb)
                b = oracle_mod.dequantize_value(2 * MAX - q, bins, mb)
                assert a == -b


def test_dequantize_binary32_steps(oracle_mod):
    # (q - MAX) / MAX and the product with max1 are each one binary32 rounding:
    # for bins = 32 (MAX = 15), q = 16, max1 = 0.1 (fp16 0.0999755859375):
    # 1/15 -> binary32 0x3D888889; times max1 rounded once more.
    one_15 = np.float32(1.0) / np.float32(15.0)
    assert one_15.view(np.uint32) == 0x3D888889
    expect = np.float32(one_15 * np.float32(np.float16(0.1)))
    got = np.float32(oracle_mod.dequantize_value(16, 32, int(np.float16(0.1).view(np.uint16))))
    assert got == expect


def test_layerwise_bins_bound_symbols(oracle_mod, synth_mod):
    w = synth_mod.WORKLOADS["tiny"]
    k, v = synth_mod.generate(w)
    sym, max1 = oracle_mod.quantize(k, v, w.bins_k, w.bins_v)
    for kv, x in enumerate((k, v)):
        for l in range(w.L):
            MAX = w.bins_k[l] // 2 - 1
            assert sym[kv, l].max() <= 2 * MAX
            # max1 is amax |x| over the channels of each token
            ref = np.abs(x[l].astype(np.float32)).max(axis=1).astype(np.float16)
            assert (max1[kv, l] == ref.view(np.uint16)).all()
