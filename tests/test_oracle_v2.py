"""Pins for the oracle's format 2 (side information as symbol counts): the
alphabet against what quantisation can produce, hand-checked records, the
record <-> counts round trip, F2 against format 1's F, the record layout, and
format 2 decoding to exactly format 1's values (both are lossless codes of the
same symbols, [CG §2.3(2)], [CG §2.4])."""
import numpy as np
import pytest


def _rand_kv(rng, L, T, C_):
    k = (rng.standard_normal((L, T, C_)) * rng.lognormal(0, 0.5, (1, 1, C_))).astype(np.float16)
    v = (rng.standard_normal((L, T, C_)) * 0.7).astype(np.float16)
    return k, v


@pytest.mark.parametrize("bins", [4, 5, 7, 8, 16, 31, 32, 100, 255, 256])
def test_alphabet_is_the_range_quantisation_produces(oracle_mod, bins):
    A = oracle_mod.alphabet_v2(bins)
    MAX = bins // 2 - 1
    assert A == 2 * MAX + 1
    # the extreme values of a group map to 0 and 2 MAX = A - 1
    x = np.array([-3.0, 3.0, 0.5, 0.0], np.float16)
    q, _ = oracle_mod.quantize_group(x, bins)
    assert int(q.min()) == 0 and int(q.max()) == A - 1


@pytest.mark.parametrize("counts,rec", [
    ([1, 5, 2], [1, 1, 2]),                # mode 1 first, then n_0, n_2
    ([2, 2, 0], [0, 2, 0]),                # tie: the smaller symbol is the mode
    ([0, 0, 7, 0, 0], [2, 0, 0, 0, 0]),    # one symbol only
    ([3, 0, 0, 0, 4], [4, 3, 0, 0, 0]),    # mode last
])
def test_record_hand_examples(oracle_mod, counts, rec):
    assert oracle_mod.record_from_counts(counts).tolist() == rec
    assert oracle_mod.counts_from_record(rec, sum(counts)).tolist() == counts


def test_record_rejects_large_non_mode_count(oracle_mod):
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.record_from_counts([300, 300, 0])     # only possible beyond 256 tokens
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.counts_from_record([3, 0, 0], 5)      # mode byte outside the alphabet
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.counts_from_record([0, 9, 9], 10)     # stored counts exceed the tokens


def test_record_round_trip_random(oracle_mod):
    rng = np.random.default_rng(3)
    for _ in range(300):
        A = int(rng.choice([3, 5, 7, 15, 31]))
        Tk = int(rng.integers(1, 257))
        p = rng.dirichlet(np.full(A, 0.3))
        n = rng.multinomial(Tk, p)
        rec = oracle_mod.record_from_counts(n)
        assert rec.size == A and int(rec[0]) == int(np.argmax(n))
        assert np.array_equal(oracle_mod.counts_from_record(rec, Tk), n)


def test_f2_equals_f_when_the_mode_is_the_argmax(oracle_mod):
    rng = np.random.default_rng(5)
    for _ in range(200):
        A = int(rng.choice([3, 15, 31]))
        Tk = int(rng.integers(1, 257))
        n = rng.multinomial(Tk, rng.dirichlet(np.full(A, 0.5)))
        assert np.array_equal(oracle_mod.cdf_from_counts_mode(n, Tk, int(np.argmax(n))),
                              oracle_mod.cdf_from_counts(n, Tk))


def test_record_layout_partitions_the_buffer(oracle_mod):
    L, T, C_, Tc = 3, 70, 5, 32
    bk, bv = [32, 16, 7], [8, 8, 256]
    total = oracle_mod.rec_bytes(L, T, C_, Tc, bk, bv)
    nch = -(-T // Tc)
    assert total == nch * C_ * sum(oracle_mod.alphabet_v2(b) for b in bk + bv)
    spans = []
    for k in range(nch):
        for kv, bins in ((0, bk), (1, bv)):
            for l in range(L):
                for c in range(C_):
                    spans.append((oracle_mod.rec_offset(L, C_, bk, bv, k, kv, l, c),
                                  oracle_mod.alphabet_v2(bins[l])))
    spans.sort()
    pos = 0
    for o, a in spans:
        assert o == pos
        pos += a
    assert pos == total


@pytest.mark.parametrize("L,T,C_,Tc,bk,bv", [
    (2, 64, 64, 64, [32, 16], [16, 32]),
    (3, 200, 40, 64, [32, 16, 8], [16, 16, 16]),   # ragged last chunk
    (1, 37, 24, 16, [7], [5]),                      # odd bins
])
def test_v2_decodes_to_format_1_values(oracle_mod, L, T, C_, Tc, bk, bv):
    rng = np.random.default_rng(T + C_)
    k, v = _rand_kv(rng, L, T, C_)
    r1 = oracle_mod.compress(k, v, Tc, bk, bv)
    d1k, d1v = oracle_mod.decompress(r1["packed"], r1["off"], r1["len"], r1["cdf"], r1["max1"],
                                     L, T, C_, Tc, bk, bv)
    r2 = oracle_mod.compress_v2(k, v, Tc, bk, bv)
    assert np.array_equal(r2["max1"], r1["max1"])
    d2k, d2v = oracle_mod.decompress_v2(r2["packed"], r2["off"], r2["len"], r2["rec"], r2["max1"],
                                        L, T, C_, Tc, bk, bv)
    assert np.array_equal(d2k.view(np.uint32), d1k.view(np.uint32))
    assert np.array_equal(d2v.view(np.uint32), d1v.view(np.uint32))
    # the records hold the counts of the quantised symbols
    sym, _ = oracle_mod.quantize(k, v, bk, bv)
    for kc in range(-(-T // Tc)):
        t0, t1 = kc * Tc, min(T, (kc + 1) * Tc)
        for kv, bins in ((0, bk), (1, bv)):
            for l in range(L):
                A = oracle_mod.alphabet_v2(bins[l])
                for c in range(C_):
                    o = oracle_mod.rec_offset(L, C_, bk, bv, kc, kv, l, c)
                    n = oracle_mod.counts_from_record(r2["rec"][o:o + A], t1 - t0)
                    ref = np.bincount(sym[kv, l, t0:t1, c], minlength=A)
                    assert np.array_equal(n, ref)
    # side information shrinks: A_l bytes per channel instead of 2 * max bins
    assert r2["rec"].nbytes < r1["cdf"].nbytes / 2


def test_v2_stream_sizes_near_entropy(oracle_mod):
    rng = np.random.default_rng(11)
    L, T, C_, Tc = 2, 256, 64, 256
    k, v = _rand_kv(rng, L, T, C_)
    bk = [32, 16]
    r2 = oracle_mod.compress_v2(k, v, Tc, bk, bk)
    sym, _ = oracle_mod.quantize(k, v, bk, bk)
    H = 0.0
    for kv in range(2):
        for l in range(L):
            for c in range(C_):
                n = np.bincount(sym[kv, l, :, c])
                p = n[n > 0] / T
                H += -(n[n > 0] * np.log2(p)).sum()
    ns = 2 * L * T
    assert r2["len"].sum() <= 1.01 * H / 8 + 4 * ns


def test_v2_rejects_chunks_over_256(oracle_mod):
    rng = np.random.default_rng(1)
    k, v = _rand_kv(rng, 1, 300, 8)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.compress_v2(k, v, 300, [16], [16])
