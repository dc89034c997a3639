"""Pins for the oracle's binary16 output (serving layouts): its float->half
rounding against IEEE round-to-nearest-even as numpy implements it (an
independent library routine), exhaustively on the round trip of every half
value, on constructed ties, and on random binary32 bit patterns across the
exponent range; and half dequantisation against numpy's conversion of the
binary32 dequantisation ([CG §2.4(2)])."""
import numpy as np


def test_every_half_round_trips(oracle_mod):
    h = np.arange(65536, dtype=np.uint32)
    exp = (h >> 10) & 0x1F
    man = h & 0x3FF
    finite = ~((exp == 31) & (man != 0))   # NaN payloads aside
    for v in h[finite][::1]:
        f = np.float32(oracle_mod.half_to_float(int(v)))
        assert oracle_mod.float_to_half(f) == int(v)


def test_ties_round_to_even(oracle_mod):
    # midpoints between consecutive halves in several binades, and in the subnormal range
    for base in [0x3C00, 0x3C01, 0x0400, 0x0001, 0x0002, 0x7BFE, 0x1234]:
        a = np.float64(np.uint16(base).view(np.float16))
        b = np.float64(np.uint16(base + 1).view(np.float16))
        mid = np.float32((a + b) / 2)
        assert float(mid) == (a + b) / 2   # the midpoint is exact in binary32
        want = base if base % 2 == 0 else base + 1
        assert oracle_mod.float_to_half(mid) == want
        assert oracle_mod.float_to_half(-mid) == want | 0x8000


def test_random_bit_patterns_match_numpy(oracle_mod):
    rng = np.random.default_rng(7)
    # exponents from far below the half subnormals to above the half maximum
    e = rng.integers(127 - 30, 127 + 17, 40000).astype(np.uint32)
    m = rng.integers(0, 1 << 23, 40000).astype(np.uint32)
    s = rng.integers(0, 2, 40000).astype(np.uint32)
    bits = (s << 31) | (e << 23) | m
    xs = bits.view(np.float32)
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.float_to_half(x) for x in xs], np.uint16)
    assert np.array_equal(got, want)


def test_special_values(oracle_mod):
    assert oracle_mod.float_to_half(np.float32(np.inf)) == 0x7C00
    assert oracle_mod.float_to_half(np.float32(-np.inf)) == 0xFC00
    assert oracle_mod.float_to_half(np.float32(0.0)) == 0
    assert oracle_mod.float_to_half(np.float32(-0.0)) == 0x8000
    assert oracle_mod.float_to_half(np.float32(1e-30)) == 0
    assert oracle_mod.float_to_half(np.float32(70000.0)) == 0x7C00
    assert (oracle_mod.float_to_half(np.float32(np.nan)) & 0x7C00) == 0x7C00


def test_half_dequantisation_is_rounded_binary32(oracle_mod):
    rng = np.random.default_rng(9)
    L, T, C_ = 2, 40, 24
    k = (rng.standard_normal((L, T, C_)) * 3).astype(np.float16)
    v = (rng.standard_normal((L, T, C_)) * 1e-3).astype(np.float16)   # small values: half subnormals
    bk, bv = [32, 7], [16, 4]
    sym, max1 = oracle_mod.quantize(k, v, bk, bv)
    fk, fv = oracle_mod.dequantize(sym, max1, bk, bv)
    hk, hv = oracle_mod.dequantize_half(sym, max1, bk, bv)
    assert np.array_equal(hk, fk.astype(np.float16).view(np.uint16))
    assert np.array_equal(hv, fv.astype(np.float16).view(np.uint16))
