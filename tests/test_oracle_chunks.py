"""A chunk coded alone by the oracle is exactly that chunk's block of the
whole tensor's outputs (the premise of the full-size GPU checks, which code
sampled chunks alone): on 600 tokens of the 4096-token workload, three chunks
with a ragged last one of 88 tokens, in all three formats."""
import hashlib

import numpy as np
import pytest

import oracle_chunks


@pytest.mark.parametrize("fmt", [1, 2, 3])
def test_chunk_alone_is_block_of_whole(oracle_mod, synth_mod, fmt):
    w = synth_mod.WORKLOADS["ctx4096"]
    T = 600
    L, C_, Tc, bk, bv = w.L, w.C, w.chunk_tokens, w.bins_k, w.bins_v
    k, v = synth_mod.generate(w, T=T)
    if fmt == 1:
        r = oracle_mod.compress(k, v, Tc, bk, bv)
        side = r["cdf"]
        dk, dv = oracle_mod.decompress(r["packed"], r["off"], r["len"], r["cdf"], r["max1"], L, T, C_, Tc, bk, bv)
    elif fmt == 2:
        r = oracle_mod.compress_v2(k, v, Tc, bk, bv)
        side = r["rec"]
        dk, dv = oracle_mod.decompress_v2(r["packed"], r["off"], r["len"], r["rec"], r["max1"], L, T, C_, Tc, bk, bv)
    else:
        r = oracle_mod.compress_v3(k, v, Tc, bk, bv)
        side = oracle_mod.v3_to_records(r["side"], L, T, C_, Tc, bk, bv)
        dk, dv = oracle_mod.decompress_v3(r["packed"], r["len"], r["side"], r["max1"], L, T, C_, Tc, bk, bv)
    for kc in range(3):
        ref = oracle_chunks.code_chunk("ctx4096", kc, fmt, T=T)
        t0, t1 = kc * Tc, min(T, (kc + 1) * Tc)
        assert np.array_equal(r["max1"][:, :, t0:t1], ref["max1"])
        if fmt == 1:
            g0 = oracle_mod.cdf_offset(L, C_, max(bk), max(bv), kc, 0, 0, 0)
        else:
            g0 = oracle_mod.rec_offset(L, C_, bk, bv, kc, 0, 0, 0)
        assert np.array_equal(side[g0:g0 + ref["side"].size], ref["side"])
        s0 = oracle_mod.stream_id(L, T, Tc, kc, 0, 0, 0)
        ns = 2 * L * (t1 - t0)
        assert np.array_equal(r["len"][s0:s0 + ns], ref["len"])
        b0, b1 = int(r["off"][s0]), int(r["off"][s0 + ns])
        assert np.array_equal(r["packed"][b0:b1], ref["packed"])
        h = hashlib.sha256()
        h.update(np.ascontiguousarray(dk[:, t0:t1]).tobytes())
        h.update(np.ascontiguousarray(dv[:, t0:t1]).tobytes())
        assert h.hexdigest() == ref["out_sha256"]
    assert kc == 2 and t1 - t0 == 88
