"""Pins for the oracle's range coder ([CG §1.2(3)] arithmetic coding,
[CG §2.4(1)] GPU decoding; constants from the codec specification).

- hand-traced streams (tests/golden/coder_hand_traces.txt);
- exhaustive brute force: every string of length 1..6 over 3 symbols;
- a big-integer restatement of the coder: the interval's lower end kept at
  full precision, so the output is the top bytes of an exact sum and no carry
  rule is needed -- it must agree byte for byte with the oracle's 32-bit
  state and carry walk;
- information bounds: 8 * len >= sum -log2(f/M) and
  8 * (len - 1) < sum -log2(f/M) + n * -log2(1 - 2^-8);
- the decoder reads exactly len + 3 bytes of a valid stream.
"""
import itertools
import math

import numpy as np
import pytest

from conftest import read_golden

M = 65536


def _row_freq(row, s):
    A = len(row)
    hi = M if s + 1 >= A else int(row[s + 1])
    return hi - int(row[s])


def bigint_encode(syms, rows):
    """Coder of the specification with the lower end LOW as an exact integer
    scaled by 2^(8*shifts): emitted bytes are the top bytes of LOW."""
    LOW, rng, shifts = 0, 0xFFFFFFFF, 0
    for s, row in zip(syms, rows):
        r = rng >> 16
        LOW += r * int(row[s])
        rng = r * _row_freq(row, s)
        while rng < (1 << 24):
            LOW <<= 8
            rng <<= 8
            shifts += 1
    V = LOW + 0x00FFFFFF
    assert V < 1 << (32 + 8 * shifts)
    return (V >> 24).to_bytes(shifts + 1, "big")


def ideal_bits(syms, rows):
    return sum(-math.log2(_row_freq(row, s) / M) for s, row in zip(syms, rows))


def _check_bounds(data, syms, rows):
    n = len(syms)
    ideal = ideal_bits(syms, rows)
    assert 8 * len(data) >= ideal - 1e-9
    assert 8 * (len(data) - 1) < ideal + n * -math.log2(1 - 2.0 ** -8) + 1e-6


@pytest.mark.parametrize("row", read_golden("coder_hand_traces.txt"), ids=lambda r: r[0])
def test_hand_traces(oracle_mod, row):
    cdf = np.array([int(t) for t in row[1].split()], np.uint16)
    syms = [int(t) for t in row[2].split()]
    expect = bytes.fromhex(row[3])
    got = oracle_mod.encode_stream(syms, cdf)
    assert got == expect
    back, used, st = oracle_mod.decode_stream(got, len(syms), cdf)
    assert list(back) == syms and st == 0 and used == len(got) + 3


CDFS_3 = {
    "uniform": [0, 21845, 43690],
    "skew_mid": [0, 1, 65535],
    "skew_low": [0, 65534, 65535],
    "random": [0, 9000, 50001],
}


@pytest.mark.parametrize("name", list(CDFS_3))
def test_exhaustive_three_symbols(oracle_mod, name):
    cdf = np.array(CDFS_3[name], np.uint16)
    seen = {}
    for n in range(1, 7):
        for syms in itertools.product(range(3), repeat=n):
            data = oracle_mod.encode_stream(list(syms), cdf)
            back, used, st = oracle_mod.decode_stream(data, n, cdf)
            assert tuple(back) == syms, (syms, data.hex())
            assert st == 0 and used == len(data) + 3
            assert data == bigint_encode(syms, [cdf] * n)
            _check_bounds(data, syms, [cdf] * n)
            key = (n, data)
            assert key not in seen, f"{syms} and {seen.get(key)} share a stream"
            seen[key] = syms
    assert len(seen) == sum(3 ** n for n in range(1, 7)) == 1092


def _random_cdf(rng, A):
    f = rng.dirichlet(np.full(A, rng.uniform(0.05, 3.0)))
    n = rng.multinomial(4096, f).astype(np.uint32)
    return n


def test_bigint_agreement_random(oracle_mod):
    """Random skewed models and strings, including carry chains."""
    rng = np.random.default_rng(11)
    carries = chains = 0
    for trial in range(400):
        A = int(rng.choice([2, 3, 8, 16, 32, 256]))
        n = int(rng.integers(1, 300))
        rows = []
        for _ in range(n):
            cnt = _random_cdf(rng, A)
            rows.append(oracle_mod.cdf_from_counts(cnt, int(cnt.sum())))
        rows = np.array(rows, np.uint16)
        # draw symbols from the model so streams look like real data; add some
        # improbable symbols to force long renormalisations
        f = np.diff(np.append(rows.astype(np.int64), np.full((n, 1), M), axis=1), axis=1)
        syms = [int(rng.choice(A, p=f[i] / M)) if rng.random() > 0.05 else int(rng.integers(0, A))
                for i in range(n)]
        data = oracle_mod.encode_stream(syms, rows)
        assert data == bigint_encode(syms, rows)
        _check_bounds(data, syms, rows)
        back, used, st = oracle_mod.decode_stream(data, n, rows)
        assert list(back) == syms and st == 0 and used == len(data) + 3
        # count streams where a carry ran through a 0xFF byte (seen as a
        # 0x00 byte right after a byte that received the carry)
        carries += data.count(b"\x00")
        chains += any(data[i] == 0 and data[i + 1] == 0 for i in range(len(data) - 1))
    assert carries > 0


def test_carry_through_ff_chain(oracle_mod):
    """Search strings until the big-integer model shows a carry that crossed
    at least one 0xFF byte (an emitted 0xFF later turned into 0x00), and check
    the oracle on each of them."""
    rng = np.random.default_rng(5)
    cdf = np.array([0, 65280], np.uint16)  # f0 = 65280, f1 = 256
    found = 0
    for _ in range(20000):
        n = int(rng.integers(2, 12))
        syms = list(rng.integers(0, 2, size=n))
        # bytes emitted so far by a carry-less replay, to see FF -> 00 flips
        data = oracle_mod.encode_stream(syms, cdf)
        ref = bigint_encode(syms, [cdf] * n)
        assert data == ref
        raw = _emitted_before_carries(syms, cdf)
        if any(a == 0xFF and b == 0x00 for a, b in zip(raw, data)):
            found += 1
            back, used, st = oracle_mod.decode_stream(data, n, cdf)
            assert list(back) == syms and st == 0
    assert found > 0


def _emitted_before_carries(syms, cdf):
    """Bytes as first emitted (32-bit low, carries dropped)."""
    low, rng, out = 0, 0xFFFFFFFF, []
    for s in syms:
        r = rng >> 16
        low = (low + r * int(cdf[s])) & 0xFFFFFFFF
        rng = r * _row_freq(cdf, s)
        while rng < (1 << 24):
            out.append(low >> 24)
            low = (low << 8) & 0xFFFFFFFF
            rng <<= 8
    out.append(((low + 0xFFFFFF) & 0xFFFFFFFF) >> 24)
    return out


def test_empty_stream_is_one_flush_byte(oracle_mod):
    cdf = np.array([0, 32768], np.uint16)
    data = oracle_mod.encode_stream([], cdf)
    assert data == b"\x00"
    back, used, st = oracle_mod.decode_stream(data, 0, cdf)
    assert st == 0 and used == 4


def test_worst_case_length_fits_scratch(oracle_mod):
    """Least probable symbol everywhere (f = 1, A = 256): the stream stays
    within 2*C + 8 bytes, the per-stream bound used for scratch sizing."""
    A = 256
    cnt = np.zeros(A, np.uint32)
    cnt[0] = 256
    row = oracle_mod.cdf_from_counts(cnt, 256)
    for C in (1, 7, 64, 1024):
        data = oracle_mod.encode_stream([A - 1] * C, row)
        assert len(data) <= 2 * C + 8
        assert data == bigint_encode([A - 1] * C, [row] * C)


def test_truncated_stream_flags_or_differs(oracle_mod):
    rng = np.random.default_rng(3)
    cdf = oracle_mod.cdf_from_counts([50, 100, 80, 26], 256)
    syms = list(rng.integers(0, 4, size=200))
    data = oracle_mod.encode_stream(syms, cdf)
    back, used, st = oracle_mod.decode_stream(data[:-5], len(syms), cdf)
    assert st != 0 or list(back) != syms
