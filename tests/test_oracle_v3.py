"""Pins for the oracle's format 3 (compact count records): the side buffer
byte for byte on a hand-built example, its sizes, the round trip against
format 2's records on random valid records, the streams identical to format
2's, decompression from the lengths alone, the delta, and every kind of
malformed buffer rejected."""
import numpy as np
import pytest


def _le(x, n):
    return list(int(x).to_bytes(n, "little"))


def test_hand_built_side_buffer(oracle_mod):
    """One layer, C = 2, T = 4, Tc = 4, bins 8 (A = 7) for K and V: one chunk,
    slices K (s = 0) and V (s = 1), four records. Format 2 records (mode, then
    the counts of the other symbols in increasing order):
      K c0: mode 3, counts of 0,1,2,4,5,6 = 0,1,0,0,0,0   -> bits {1}, V: 1
      K c1: mode 3, counts = 0,0,1,1,1,0                   -> bits {2,4,5}, V: 1,1,1
      V c0: mode 0, counts of 1..6 = 0,0,0,0,0,0           -> bits {}, V: -
      V c1: mode 6, counts of 0..5 = 2,0,0,0,0,0           -> bits {0}, V: 2
    O = [0, 4, 5]; offM = 24, offB = 28 (24 + 4), offV = 44."""
    rec = np.array([3, 0, 1, 0, 0, 0, 0,
                    3, 0, 0, 1, 1, 1, 0,
                    0, 0, 0, 0, 0, 0, 0,
                    6, 2, 0, 0, 0, 0, 0], np.uint8)
    L, T, C_, Tc, bins = 1, 4, 2, 4, [8]
    assert oracle_mod.v3_fixed_bytes(L, T, C_, Tc) == 44
    side = oracle_mod.records_to_v3(rec, L, T, C_, Tc, bins, bins)
    want = (_le(0, 8) + _le(4, 8) + _le(5, 8) + [3, 3, 0, 6]
            + _le(1 << 1, 4) + _le((1 << 2) | (1 << 4) | (1 << 5), 4) + _le(0, 4) + _le(1 << 0, 4)
            + [1, 1, 1, 1, 2])
    assert list(side) == want
    assert np.array_equal(oracle_mod.v3_to_records(side, L, T, C_, Tc, bins, bins), rec)


def _random_records(rng, L, T, C_, Tc, bk, bv, oracle_mod):
    """Valid format 2 records: counts summing to each chunk's tokens."""
    rec = np.zeros(oracle_mod.rec_bytes(L, T, C_, Tc, bk, bv), np.uint8)
    nch = -(-T // Tc)
    for kc in range(nch):
        Tk = min(Tc, T - kc * Tc)
        for kv, bins in enumerate((bk, bv)):
            for l in range(L):
                A = oracle_mod.alphabet_v2(bins[l])
                for c in range(C_):
                    p = rng.dirichlet(np.full(A, rng.uniform(0.05, 2.0)))
                    n = rng.multinomial(Tk, p)
                    o = oracle_mod.rec_offset(L, C_, bk, bv, kc, kv, l, c)
                    rec[o:o + A] = oracle_mod.record_from_counts(n)
    return rec


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_round_trip_and_size(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    L, T, C_, Tc = 3, 150, 12, 64
    bk, bv = [32, 16, 8], [4, 33, 16]
    rec = _random_records(rng, L, T, C_, Tc, bk, bv, oracle_mod)
    side = oracle_mod.records_to_v3(rec, L, T, C_, Tc, bk, bv)
    assert np.array_equal(oracle_mod.v3_to_records(side, L, T, C_, Tc, bk, bv), rec)
    # size = fixed part + one byte per nonzero count byte of the records
    nonzero = 0
    nch = -(-T // Tc)
    for kc in range(nch):
        for kv, bins in enumerate((bk, bv)):
            for l in range(L):
                A = oracle_mod.alphabet_v2(bins[l])
                for c in range(C_):
                    o = oracle_mod.rec_offset(L, C_, bk, bv, kc, kv, l, c)
                    nonzero += int(np.count_nonzero(rec[o + 1:o + A]))
    assert side.size == oracle_mod.v3_fixed_bytes(L, T, C_, Tc) + nonzero
    assert side.size <= oracle_mod.v3_max_bytes(L, T, C_, Tc, bk, bv)


def test_limits(oracle_mod):
    assert oracle_mod.v3_fixed_bytes(1, 600, 8, 300) == 0          # chunks over 256 tokens
    assert oracle_mod.v3_max_bytes(1, 64, 8, 64, [64], [16]) == 0  # A = 63 > 32 bits


@pytest.mark.parametrize("G", [1, 10])
def test_streams_equal_format2_and_decompress_from_lengths(oracle_mod, synth_mod, G):
    w = synth_mod.WORKLOADS["tiny"]
    k, v = synth_mod.generate(w)
    L, T, C_ = k.shape
    Tc = w.chunk_tokens
    r2 = oracle_mod.compress_ex(k, v, Tc, w.bins_k, w.bins_v, fmt=2, group=G)
    r3 = oracle_mod.compress_v3(k, v, Tc, w.bins_k, w.bins_v, group=G)
    for key in ("max1", "packed", "len", "off"):
        assert np.array_equal(r2[key], r3[key]), key
    assert np.array_equal(oracle_mod.v3_to_records(r3["side"], L, T, C_, Tc, w.bins_k, w.bins_v), r2["rec"])
    ok, ov = oracle_mod.decompress_v3(r3["packed"], r3["len"], r3["side"], r3["max1"], L, T, C_, Tc,
                                      w.bins_k, w.bins_v, group=G)
    rk, rv = oracle_mod.decompress_ex(r2["packed"], r2["off"], r2["len"], r2["rec"], r2["max1"], L, T, C_, Tc,
                                      w.bins_k, w.bins_v, fmt=2, group=G)
    assert np.array_equal(ok.view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(ov.view(np.uint32), rv.view(np.uint32))
    assert r3["side"].size < r2["rec"].size


def test_malformed_buffers_rejected(oracle_mod):
    rec = np.array([3, 0, 1, 0, 0, 0, 0,
                    3, 0, 0, 1, 1, 1, 0,
                    0, 0, 0, 0, 0, 0, 0,
                    6, 2, 0, 0, 0, 0, 0], np.uint8)
    args = (1, 4, 2, 4, [8], [8])
    good = oracle_mod.records_to_v3(rec, *args)
    offM, offB, offV = 24, 28, 44

    def bad(mutate):
        s = good.copy()
        mutate(s)
        with pytest.raises(oracle_mod.OracleError):
            oracle_mod.v3_to_records(s, *args)

    def set_u32(s, at, x):
        s[at:at + 4] = np.frombuffer(int(x).to_bytes(4, "little"), np.uint8)

    bad(lambda s: s.__setitem__(offM, 7))                       # mode outside A = 7
    bad(lambda s: set_u32(s, offB, (1 << 1) | (1 << 3)))        # the mode's own bit
    bad(lambda s: set_u32(s, offB, (1 << 1) | (1 << 7)))        # a bit at A
    bad(lambda s: s.__setitem__(offV, 0))                       # a zero count under a set bit
    bad(lambda s: s.__setitem__(8, 6))                          # O[1] past O[2]
    bad(lambda s: s.__setitem__(16, 9))                         # O[2] past the buffer
    bad(lambda s: s.__setitem__(0, 1))                          # O[0] not 0
    with pytest.raises(oracle_mod.OracleError):                 # truncated
        oracle_mod.v3_to_records(good[:-1], *args)
    with pytest.raises(oracle_mod.OracleError):                 # shorter than its fixed part
        oracle_mod.v3_to_records(good[:40], *args)
