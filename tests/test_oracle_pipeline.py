"""Whole-tensor pins for the oracle: lossless coding, the quantisation error
bound, size against the empirical entropy, chunk independence and the packed
layout ([CG §2.3(1)-(3)], [CG §2.4(1)-(2)])."""
import math

import numpy as np
import pytest


def _ragged_case(rng):
    L, T, C, Tc = 3, 150, 40, 64  # chunks of 64, 64 and a ragged 22
    k = (rng.standard_normal((L, T, C)) * rng.lognormal(0, 0.5, size=(1, 1, C))).astype(np.float16)
    v = (rng.standard_t(3, size=(L, T, C))).astype(np.float16)
    k[1, 5] = 0.0  # an all-zero group
    bins_k = [32, 16, 8]
    bins_v = [4, 16, 255]  # A_V = 255 differs from A_K = 32
    return k, v, Tc, bins_k, bins_v


def _cases(synth_mod):
    rng = np.random.default_rng(42)
    w = synth_mod.WORKLOADS["tiny"]
    k, v = synth_mod.generate(w)
    yield "tiny", k, v, w.chunk_tokens, list(w.bins_k), list(w.bins_v)
    yield ("ragged",) + _ragged_case(rng)
    u = synth_mod.WORKLOADS["uniform"]
    k, v = synth_mod.generate(u, T=96)
    yield "uniform", k[:4, :, :128].copy(), v[:4, :, :128].copy(), 32, list(u.bins_k[:4]), list(u.bins_v[:4])


def test_round_trip_and_bounds(oracle_mod, synth_mod):
    for name, k, v, Tc, bk, bv in _cases(synth_mod):
        L, T, C = k.shape
        r = oracle_mod.compress(k, v, Tc, bk, bv)
        sym, max1 = oracle_mod.quantize(k, v, bk, bv)
        # lossless entropy coding: decode returns exactly the quantised symbols
        dec, st = oracle_mod.decode(r["packed"], r["off"], r["len"], r["cdf"], L, T, C, Tc,
                                    r["A_k"], r["A_v"])
        assert st == 0 and (dec == sym).all(), name
        # dequantised output obeys the error bound per group
        ok, ov = oracle_mod.decompress(r["packed"], r["off"], r["len"], r["cdf"], r["max1"],
                                       L, T, C, Tc, bk, bv)
        for kv, x, out, bins in ((0, k, ok, bk), (1, v, ov, bv)):
            m1 = max1[kv].view(np.float16).astype(np.float64)  # [L, T]
            MAX = (np.asarray(bins) // 2 - 1).astype(np.float64)[:, None]
            bound = m1 / (2 * MAX) + np.spacing(max1[kv].view(np.float16)).astype(np.float64)
            err = np.abs(out.astype(np.float64) - x.astype(np.float64)).max(axis=2)
            assert (err <= bound).all(), name
        # packed layout: off is the exclusive scan of len
        assert r["off"][0] == 0
        assert (np.diff(r["off"].astype(np.int64)) == r["len"]).all()
        assert r["packed"].size == int(r["off"][-1])


def test_size_near_empirical_entropy(oracle_mod, synth_mod):
    """sum len <= 1.01 * H_emp / 8 + 4 bytes per stream, where H_emp uses the
    chunk's own symbol counts per (kv, layer, channel)."""
    for name, k, v, Tc, bk, bv in _cases(synth_mod):
        L, T, C = k.shape
        r = oracle_mod.compress(k, v, Tc, bk, bv)
        sym, _ = oracle_mod.quantize(k, v, bk, bv)
        H = 0.0
        for c0 in range(0, T, Tc):
            blk = sym[:, :, c0:c0 + Tc, :]
            Tk = blk.shape[2]
            for kv in range(2):
                for l in range(L):
                    for c in range(C):
                        n = np.bincount(blk[kv, l, :, c])
                        n = n[n > 0].astype(np.float64)
                        H += -(n * np.log2(n / Tk)).sum()
        ns = 2 * L * T
        total = int(r["off"][-1])
        assert total <= 1.01 * H / 8 + 4 * ns, (name, total, H / 8)


def test_chunks_are_independent(oracle_mod, synth_mod):
    """Chunk k of the full output equals the output of chunk k coded alone."""
    rng = np.random.default_rng(9)
    k, v, Tc, bk, bv = _ragged_case(rng)
    L, T, C = k.shape
    full = oracle_mod.compress(k, v, Tc, bk, bv)
    A_k, A_v = full["A_k"], full["A_v"]
    per_chunk_cdf = L * C * (A_k + A_v)
    for ci, t0 in enumerate(range(0, T, Tc)):
        t1 = min(T, t0 + Tc)
        part = oracle_mod.compress(k[:, t0:t1].copy(), v[:, t0:t1].copy(), Tc, bk, bv)
        s0 = oracle_mod.stream_id(L, T, Tc, ci, 0, 0, 0)
        s1 = s0 + 2 * L * (t1 - t0)
        assert (full["len"][s0:s1] == part["len"]).all()
        b0, b1 = int(full["off"][s0]), int(full["off"][s1])
        assert full["packed"][b0:b1].tobytes() == part["packed"].tobytes()
        assert (full["cdf"][ci * per_chunk_cdf:(ci + 1) * per_chunk_cdf] == part["cdf"]).all()
        assert (full["max1"][:, :, t0:t1] == part["max1"]).all()


def test_each_stream_is_its_tokens_channels(oracle_mod):
    """Stream sid(k, kv, l, t) is the coding of q[kv][l][t][0..C-1] with the
    CDF rows of (k, kv, l, c) in channel order."""
    rng = np.random.default_rng(4)
    k, v, Tc, bk, bv = _ragged_case(rng)
    L, T, C = k.shape
    r = oracle_mod.compress(k, v, Tc, bk, bv)
    sym, _ = oracle_mod.quantize(k, v, bk, bv)
    A = (r["A_k"], r["A_v"])
    for ci, kv, l, tl in [(0, 0, 0, 0), (1, 1, 2, 63), (2, 0, 1, 21), (2, 1, 2, 0)]:
        t = ci * Tc + tl
        sid = oracle_mod.stream_id(L, T, Tc, ci, kv, l, tl)
        o = oracle_mod.cdf_offset(L, C, A[0], A[1], ci, kv, l, 0)
        rows = r["cdf"][o:o + C * A[kv]].reshape(C, A[kv])
        data = oracle_mod.encode_stream(sym[kv, l, t], rows)
        b = int(r["off"][sid])
        assert r["packed"][b:b + r["len"][sid]].tobytes() == data


def test_stream_ids_cover_everything_once(oracle_mod):
    L, T, Tc = 3, 150, 64
    ids = set()
    for ci in range(math.ceil(T / Tc)):
        Tk = min(Tc, T - ci * Tc)
        for kv in range(2):
            for l in range(L):
                for tl in range(Tk):
                    ids.add(oracle_mod.stream_id(L, T, Tc, ci, kv, l, tl))
    assert ids == set(range(2 * L * T))


def test_capacity_shortfall_reported(oracle_mod, synth_mod):
    w = synth_mod.WORKLOADS["tiny"]
    k, v = synth_mod.generate(w)
    sym, _ = oracle_mod.quantize(k, v, w.bins_k, w.bins_v)
    cdf = oracle_mod.calculate_cdf(sym, w.chunk_tokens, 32, 32)
    packed, ln, off, st = oracle_mod.encode(sym, cdf, w.chunk_tokens, 32, 32, capacity=100)
    assert st == oracle_mod.ERR_CAPACITY
    assert int(off[-1]) > 100 and packed.size == 100
    full, ln2, off2, st2 = oracle_mod.encode(sym, cdf, w.chunk_tokens, 32, 32)
    assert st2 == 0 and (ln == ln2).all() and (off == off2).all()
    assert packed.tobytes() == full[:100].tobytes()


@pytest.mark.parametrize("T", [1, 2, 255, 256, 257])
def test_token_count_edges(oracle_mod, T):
    rng = np.random.default_rng(T)
    k = rng.standard_normal((2, T, 24)).astype(np.float16)
    v = rng.standard_normal((2, T, 24)).astype(np.float16)
    r = oracle_mod.compress(k, v, 256, [16, 8], [16, 8])
    sym, _ = oracle_mod.quantize(k, v, [16, 8], [16, 8])
    dec, st = oracle_mod.decode(r["packed"], r["off"], r["len"], r["cdf"], 2, T, 24, 256, 16, 16)
    assert st == 0 and (dec == sym).all()
