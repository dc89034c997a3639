"""Pins for the oracle's token-locality delta (the change-based encoding of
[CG §1.2(1)], specification G): rounding max1 up to binary16 against numpy's
binary16 (an independent library routine); G = 1 reducing to the plain
quantiser; a hand-worked example whose symbols tell the closed-loop anchor
(its reconstruction) from the raw anchor and the chunk-local groups from
global ones; the zero-delta closed form; the per-row error bound; the
reduction of error on correlated tokens that motivates the method; and the
coded round trip in both formats."""
import numpy as np
import pytest


def _h(bits):
    return float(np.uint16(bits).view(np.float16))


# ---------------------------------------------------------------- half_up

def test_half_up_every_half_is_fixed(oracle_mod):
    for h in range(0, 0x7C00, 7):
        assert oracle_mod.half_up(_h(h)) == h


def test_half_up_is_the_smallest_half_above(oracle_mod):
    rng = np.random.default_rng(11)
    e = rng.integers(127 - 30, 127 + 16, 20000).astype(np.uint32)
    m = rng.integers(0, 1 << 23, 20000).astype(np.uint32)
    xs = ((e << 23) | m).view(np.float32)
    for x in xs:
        x = float(x)
        h = oracle_mod.half_up(x)
        if x > 65504.0:
            assert h == 0x7BFF
            continue
        assert _h(h) >= x
        assert h == 0 or _h(h - 1) < x


def test_floats_to_half_matches_numpy(oracle_mod):
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(50000) * np.exp(rng.uniform(-20, 11, 50000))).astype(np.float32)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle_mod.floats_to_half(x), want)


# ---------------------------------------------------------------- QA / QD / DD

def test_group_of_one_is_plain_quantisation(oracle_mod):
    rng = np.random.default_rng(3)
    L, T, C_ = 2, 37, 24
    k = rng.standard_normal((L, T, C_)).astype(np.float16)
    v = (rng.standard_normal((L, T, C_)) * 3).astype(np.float16)
    sym, max1 = oracle_mod.quantize_delta(k, v, 16, 1, [32, 8], [16, 256])
    s0, m0 = oracle_mod.quantize(k, v, [32, 8], [16, 256])
    assert np.array_equal(sym, s0) and np.array_equal(max1, m0)
    ok, ov = oracle_mod.dequantize_delta(sym, max1, 16, 1, [32, 8], [16, 256])
    pk, pv = oracle_mod.dequantize(s0, m0, [32, 8], [16, 256])
    assert np.array_equal(ok.view(np.uint32), pk.view(np.uint32))
    assert np.array_equal(ov.view(np.uint32), pv.view(np.uint32))


def _hand_case():
    # one layer, C = 4, bins 8 (MAX = 3), chunks of 3 tokens, groups of 2:
    # chunk 0 = tokens 0 (anchor), 1 (delta), 2 (anchor); chunk 1 = token 3 (anchor)
    k = np.array([[[1.0, -0.5, 0.25, 0.0],
                   [1.5, -0.5, 0.0, 0.125],
                   [2.0, 0.0, 0.0, 0.0],
                   [2.0, 1.0, 0.0, 0.0]]], np.float16)
    return k


def test_hand_worked_example(oracle_mod):
    """Worked by hand from the specification, binary32 step by step.

    token 0 (anchor): max1 = 1, factor = 3, y = 6, 1.5, 3.75, 3 -> q = 6, 2, 4, 3;
      a^ = 1, -1/3, 1/3, 0 (binary32: -0.33333334, 0.33333334).
    token 1: d = 0.5, -0.16666666 (exact), -0.33333334, 0.125 -> max1 = 0.5,
      factor = 6; d*factor = 3, -0.99999994, -2 (rounded), 0.75;
      y = 6, 2 (2 + 2^-24 rounds down), 1, 3.75 -> q = 6, 2, 1, 4.
      (Deltas against the raw anchor would give q = 6, 3, 2, 4.)
      x^ = 1.5, -0.5 (rounded), 0, 0.16666667.
    token 2: an anchor again (tl = 2): plain Q.
    token 3: first token of chunk 1, so an anchor although t = 3 is odd:
      max1 = 2 (as a delta from token 2 it would be 1)."""
    k = _hand_case()
    bins = [8]
    sym, max1 = oracle_mod.quantize_delta(k, k, 3, 2, bins, bins)
    assert list(sym[0, 0, 0]) == [6, 2, 4, 3]
    assert max1[0, 0, 0] == 0x3C00
    assert list(sym[0, 0, 1]) == [6, 2, 1, 4]
    assert max1[0, 0, 1] == 0x3800
    q2, m2 = oracle_mod.quantize_group(k[0, 2], 8)
    assert np.array_equal(sym[0, 0, 2], q2) and max1[0, 0, 2] == m2
    q3, m3 = oracle_mod.quantize_group(k[0, 3], 8)
    assert np.array_equal(sym[0, 0, 3], q3) and max1[0, 0, 3] == m3 == 0x4000
    ok, _ = oracle_mod.dequantize_delta(sym, max1, 3, 2, bins, bins)
    want1 = np.array([1.5, -0.5, 0.0, np.float32(1) / np.float32(6)], np.float32)
    assert want1[3] == np.float32(0.16666667)
    assert np.array_equal(ok[0, 1].view(np.uint32), want1.view(np.uint32))


def test_zero_delta_rows(oracle_mod):
    """bins 4 (MAX = 1): an anchor reconstructs to exactly -max1, 0 or max1,
    all binary16 values; rows equal to that reconstruction have d = 0, so
    max1 = 0, every symbol is MAX and x^ is the reconstruction exactly."""
    rng = np.random.default_rng(5)
    L, T, C_, Tc, G = 1, 8, 16, 8, 4
    x = rng.standard_normal((L, T, C_)).astype(np.float16)
    s0, m0 = oracle_mod.quantize(x[:, :1], x[:, :1], [4])
    a, _ = oracle_mod.dequantize(s0, m0, [4])
    assert set(np.unique(np.abs(a))) <= {0.0, float(_h(m0[0, 0, 0]))}
    x[:, 1:G] = a.astype(np.float16)
    sym, max1 = oracle_mod.quantize_delta(x, x, Tc, G, [4])
    assert (max1[0, 0, 1:G] == 0).all() and (sym[0, 0, 1:G] == 1).all()
    ok, _ = oracle_mod.dequantize_delta(sym, max1, Tc, G, [4])
    assert np.array_equal(ok[0, 1:G], np.repeat(a[0], G - 1, axis=0))


def _correlated(rng, L, T, C_, rho=0.995, scale=2.0):
    """Tokens that change slowly: an AR(1) walk around per-channel offsets."""
    off = rng.standard_normal((L, 1, C_)) * scale
    x = np.empty((L, T, C_))
    x[:, 0] = rng.standard_normal((L, C_))
    for t in range(1, T):
        x[:, t] = rho * x[:, t - 1] + np.sqrt(1 - rho * rho) * rng.standard_normal((L, C_))
    return (x * 0.3 + off).astype(np.float16)


@pytest.mark.parametrize("G,bins", [(2, 8), (10, 32), (5, 16), (64, 4)])
def test_error_bound_per_row(oracle_mod, G, bins):
    """|x - x^| <= max1/(2 MAX) plus binary32 rounding of the delta and the
    sum, on every element; anchors equal plain quantisation. Against the raw
    anchor instead of its reconstruction the anchor's own error would add
    up to max1_anchor/(2 MAX), far above this bound here."""
    rng = np.random.default_rng(G * 100 + bins)
    L, T, C_, Tc = 2, 150, 32, 64
    k = _correlated(rng, L, T, C_)
    v = _correlated(rng, L, T, C_, rho=0.9)
    sym, max1 = oracle_mod.quantize_delta(k, v, Tc, G, [bins] * L)
    ok, ov = oracle_mod.dequantize_delta(sym, max1, Tc, G, [bins] * L)
    s0, m0 = oracle_mod.quantize(k, v, [bins] * L)
    MAX = bins // 2 - 1
    tl = np.arange(T) % Tc
    anchor = (tl % G) == 0
    eps = 2.0 ** -23
    for kv, (x, out) in enumerate([(k, ok), (v, ov)]):
        assert np.array_equal(sym[kv][:, anchor], s0[kv][:, anchor])
        assert np.array_equal(max1[kv][:, anchor], m0[kv][:, anchor])
        m = max1[kv].view(np.float16).astype(np.float64)[..., None]
        xa = x.astype(np.float64)
        err = np.abs(xa - out.astype(np.float64))
        a_idx = np.arange(T) - (tl % G)
        mag = np.abs(xa) + np.abs(out.astype(np.float64)[:, a_idx]) + m
        bound = m / (2 * MAX) * (1 + 4 * eps) + 2 * eps * mag
        assert (err <= bound).all()
        if G <= 10:
            # the raw-anchor reading's extra error would not fit: on these slowly
            # changing tokens the anchors' own errors dwarf the delta rows' bound
            anchor_err = np.abs(xa - out.astype(np.float64))[:, anchor].max()
            assert anchor_err > 4 * bound[:, ~anchor].min()


def test_delta_lowers_error_on_correlated_tokens(oracle_mod):
    """The reason for the method: neighbouring tokens are similar, so deltas
    are small and, at the same bins, reconstruct with far less error."""
    rng = np.random.default_rng(9)
    L, T, C_, Tc = 2, 256, 64, 256
    k = _correlated(rng, L, T, C_, rho=0.998)
    s0, m0 = oracle_mod.quantize(k, k, [16] * L)
    p, _ = oracle_mod.dequantize(s0, m0, [16] * L)
    sym, max1 = oracle_mod.quantize_delta(k, k, Tc, 10, [16] * L)
    d, _ = oracle_mod.dequantize_delta(sym, max1, Tc, 10, [16] * L)
    xa = k.astype(np.float64)
    e_plain = np.sqrt(np.mean((xa - p) ** 2))
    e_delta = np.sqrt(np.mean((xa - d) ** 2))
    assert e_delta < 0.5 * e_plain


def test_nonfinite_and_bad_args_rejected(oracle_mod):
    x = np.zeros((1, 4, 8), np.float16)
    x[0, 1, 3] = np.inf      # a delta row (G = 2)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.quantize_delta(x, x, 4, 2, [16])
    y = np.zeros((1, 4, 8), np.float16)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.quantize_delta(y, y, 4, 0, [16])
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.quantize_delta(y, y, 4, 2, [3])


# ---------------------------------------------------------------- coded round trip

@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("G", [1, 3, 10])
def test_coded_round_trip(oracle_mod, fmt, G):
    rng = np.random.default_rng(fmt * 10 + G)
    L, T, C_, Tc = 2, 90, 16, 32
    k = _correlated(rng, L, T, C_)
    v = (rng.standard_normal((L, T, C_)) * 0.2).astype(np.float16)
    bk, bv = [32, 16], [16, 8]
    ref = oracle_mod.compress_ex(k, v, Tc, bk, bv, fmt=fmt, group=G)
    side = ref["cdf"] if fmt == 1 else ref["rec"]
    ok, ov = oracle_mod.decompress_ex(ref["packed"], ref["off"], ref["len"], side, ref["max1"],
                                      L, T, C_, Tc, bk, bv, fmt=fmt, group=G)
    sym, max1 = oracle_mod.quantize_delta(k, v, Tc, G, bk, bv)
    assert np.array_equal(ref["max1"], max1)
    wk, wv = oracle_mod.dequantize_delta(sym, max1, Tc, G, bk, bv)
    assert np.array_equal(ok.view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(ov.view(np.uint32), wv.view(np.uint32))
    if G == 1:
        plain = oracle_mod.compress(k, v, Tc, bk, bv) if fmt == 1 else oracle_mod.compress_v2(k, v, Tc, bk, bv)
        assert np.array_equal(plain["packed"], ref["packed"])
        assert np.array_equal(plain["cdf" if fmt == 1 else "rec"], side)
