"""Pins for the oracle's CDF construction ([CG §2.3(2)] calculate_cdf).

Hand-computed examples (tests/golden/cdf_hand.txt) plus invariants that any
correct 16-bit normalisation with a frequency floor of one must satisfy.
"""
import numpy as np
import pytest

from conftest import read_golden

M = 65536


def _freqs(cdf):
    c = np.append(cdf.astype(np.int64), M)
    return np.diff(c)


@pytest.mark.parametrize("row", read_golden("cdf_hand.txt"))
def test_hand_examples(oracle_mod, row):
    counts = [int(t) for t in row[0].split()]
    T = int(row[1])
    expect = [int(t) for t in row[2].split()]
    got = oracle_mod.cdf_from_counts(counts, T)
    assert list(got) == expect


def _random_counts(rng, A, T):
    kind = rng.integers(0, 4)
    if kind == 0:  # uniform multinomial
        p = np.full(A, 1.0 / A)
    elif kind == 1:  # concentrated
        p = np.zeros(A)
        p[rng.integers(0, A)] = 1.0
    elif kind == 2:  # peaked, like quantised KV around MAX
        centre = rng.integers(0, A)
        p = np.exp(-0.5 * ((np.arange(A) - centre) / rng.uniform(0.3, 4.0)) ** 2)
        p /= p.sum()
    else:  # random dirichlet
        p = rng.dirichlet(np.full(A, rng.uniform(0.05, 2.0)))
    return rng.multinomial(T, p).astype(np.uint32)


@pytest.mark.parametrize("A", [2, 3, 4, 8, 16, 31, 32, 127, 256])
def test_invariants_random(oracle_mod, A):
    rng = np.random.default_rng(1000 + A)
    for _ in range(300):
        T = int(rng.choice([1, 2, 7, 64, 255, 256, 4096, 65535]))
        n = _random_counts(rng, A, T)
        cdf = oracle_mod.cdf_from_counts(n, T)
        f = _freqs(cdf)
        assert cdf[0] == 0
        assert (f >= 1).all(), "every symbol keeps a nonzero frequency"
        assert f.sum() == M
        # proportional part: f_s - 1 = floor(n_s (M - A) / T), plus R < A on the argmax
        base = 1 + (n.astype(np.int64) * (M - A)) // T
        best = int(np.argmax(n))  # numpy argmax returns the first maximum
        extra = f - base
        assert (np.delete(extra, best) == 0).all()
        assert 0 <= extra[best] < A
        # ordering of frequencies follows ordering of counts
        N = n.astype(np.int64)
        more = N[:, None] > N[None, :]
        assert (f[:, None] >= f[None, :])[more].all()
        same = N[:, None] == N[None, :]
        assert (np.abs(f[:, None] - f[None, :]) < A)[same].all()


def test_single_symbol_takes_all_but_floor(oracle_mod):
    for A in (4, 16, 32, 256):
        for s in (0, A // 2, A - 1):
            n = np.zeros(A, np.uint32)
            n[s] = 256
            f = _freqs(oracle_mod.cdf_from_counts(n, 256))
            assert f[s] == M - (A - 1)
            assert (np.delete(f, s) == 1).all()


def test_bad_totals_rejected(oracle_mod):
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.cdf_from_counts([5, 5], 3)  # counts exceed T
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.cdf_from_counts([0, 0], 0)  # empty chunk


def test_cdf_scope_is_per_chunk_layer_channel(oracle_mod):
    """calculate_cdf over [2][L][T][C] symbols: each (chunk, kv, l, c) CDF is the
    normalisation of that column's counts over the chunk's tokens only."""
    rng = np.random.default_rng(7)
    L, T, C, Tc = 3, 150, 5, 64  # chunks of 64, 64, 22
    A_k, A_v = 8, 6
    sym = np.empty((2, L, T, C), np.uint8)
    sym[0] = rng.integers(0, A_k, size=(L, T, C))
    sym[1] = rng.integers(0, A_v, size=(L, T, C))
    cdf = oracle_mod.calculate_cdf(sym, Tc, A_k, A_v)
    assert cdf.size == 3 * L * C * (A_k + A_v)
    for k in range(3):
        t0, t1 = k * Tc, min(T, (k + 1) * Tc)
        for kv, A in ((0, A_k), (1, A_v)):
            for l in range(L):
                for c in range(C):
                    n = np.bincount(sym[kv, l, t0:t1, c], minlength=A).astype(np.uint32)
                    o = oracle_mod.cdf_offset(L, C, A_k, A_v, k, kv, l, c)
                    assert list(cdf[o:o + A]) == list(oracle_mod.cdf_from_counts(n, t1 - t0))
