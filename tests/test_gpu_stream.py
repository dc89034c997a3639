"""The chunk-pipelined streaming path: pinned host K, V in, compressed pieces
out to pinned host memory, pieces back in and decompressed. The pieces,
joined, are byte-identical to the oracle's whole-tensor output (and to one
call over the whole tensor), and the decompressed pieces equal the
single-call output row for row."""
import numpy as np
import pytest
import torch

from kv_cache_compression_cg_gb300 import shard

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T,Tc,piece_chunks", [("tiny", 64, 64, 1), ("mistral_chunk", 200, 32, 2),
                                                   ("mistral_chunk", 256, 64, 3)])
def test_stream_pieces_match_oracle_and_single_call(synth_mod, oracle_mod, name, T, Tc, piece_chunks):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    from kv_cache_compression_cg_gb300 import build, codec
    from kv_cache_compression_cg_gb300.stream import StreamingCodec
    build.build()
    w = synth_mod.WORKLOADS[name]
    k, v = synth_mod.generate(w, T=T)
    k_pin = torch.from_numpy(k).pin_memory()
    v_pin = torch.from_numpy(v).pin_memory()
    sc = StreamingCodec(w.L, T, w.C, w.bins_k, w.bins_v, chunk_tokens=Tc, piece_chunks=piece_chunks)
    pieces = sc.compress_from_host(k_pin, v_pin)  # list form, then the interleaved form
    outs, done = sc.decompress_from_host(pieces)
    done.synchronize()
    pieces, outs, done = sc.roundtrip(k_pin, v_pin)  # reuse of every buffer
    done.synchronize()
    assert sc.status() == 0
    joined = shard.assemble([hp.arrays() for hp in pieces])
    ref = oracle_mod.compress(k, v, Tc, w.bins_k, w.bins_v)
    for key in ("max1", "cdf", "packed", "len", "off"):
        assert np.array_equal(joined[key], ref[key]), key
    whole = codec.Codec(w.L, T, w.C, w.bins_k, w.bins_v, chunk_tokens=Tc)
    whole.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    rk, rv = whole.decompress()
    torch.cuda.synchronize()
    for (ok, ov), hp in zip(outs, pieces):
        assert torch.equal(ok.view(torch.int32), rk[:, hp.t0:hp.t1].view(torch.int32))
        assert torch.equal(ov.view(torch.int32), rv[:, hp.t0:hp.t1].view(torch.int32))


def test_stream_rejects_pageable_input(synth_mod):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    from kv_cache_compression_cg_gb300.stream import StreamingCodec
    w = synth_mod.WORKLOADS["tiny"]
    k, v = synth_mod.generate(w)
    sc = StreamingCodec(w.L, w.T, w.C, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens)
    with pytest.raises(ValueError):
        sc.compress_from_host(torch.from_numpy(k), torch.from_numpy(v))


@pytest.mark.parametrize("fmt", [1, 2])
def test_stream_with_delta_matches_oracle(synth_mod, oracle_mod, fmt):
    """Pieces of whole chunks code independently with the token-locality
    delta too (its groups are chunk-local): joined, they equal the oracle's
    whole-tensor output, and the decompressed pieces its values."""
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    from kv_cache_compression_cg_gb300 import build
    from kv_cache_compression_cg_gb300.stream import StreamingCodec
    build.build()
    w = synth_mod.WORKLOADS["mistral_chunk"]
    T, Tc, G = 224, 64, 10
    k, v = synth_mod.generate(w, T=T)
    k_pin = torch.from_numpy(k).pin_memory()
    v_pin = torch.from_numpy(v).pin_memory()
    sc = StreamingCodec(w.L, T, w.C, w.bins_k, w.bins_v, chunk_tokens=Tc, piece_chunks=2, fmt=fmt, group=G)
    pieces, outs, done = sc.roundtrip(k_pin, v_pin)
    done.synchronize()
    assert sc.status() == 0
    joined = shard.assemble([hp.arrays() for hp in pieces])
    ref = oracle_mod.compress_ex(k, v, Tc, w.bins_k, w.bins_v, fmt=fmt, group=G)
    side = "cdf" if fmt == 1 else "rec"
    for key in ("max1", side, "packed", "len", "off"):
        assert np.array_equal(joined[key], ref[key]), key
    wk, wv = oracle_mod.decompress_ex(ref["packed"], ref["off"], ref["len"], ref[side], ref["max1"], w.L, T, w.C,
                                      Tc, w.bins_k, w.bins_v, fmt=fmt, group=G)
    for (ok, ov), hp in zip(outs, pieces):
        assert np.array_equal(ok.cpu().numpy().view(np.uint32), wk[:, hp.t0:hp.t1].view(np.uint32))
        assert np.array_equal(ov.cpu().numpy().view(np.uint32), wv[:, hp.t0:hp.t1].view(np.uint32))


@pytest.mark.parametrize("fmt", [2, 3])
def test_stream_switches_levels_per_piece(synth_mod, oracle_mod, fmt):
    """Pieces quantised with different bins (a policy alternating two
    levels): each piece equals the oracle's compression of its tokens with its
    level's bins, and decodes to the oracle's values."""
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    from kv_cache_compression_cg_gb300 import build
    from kv_cache_compression_cg_gb300.stream import StreamingCodec
    build.build()
    w = synth_mod.WORKLOADS["mistral_chunk"]
    T, Tc = 256, 64
    k, v = synth_mod.generate(w, T=T)
    levels = [(list(w.bins_k), list(w.bins_v)), ([8] * w.L, [8] * w.L)]

    class Alternate:
        def __init__(self):
            self.calls, self.seen = 0, []

        def level_for(self, tokens):
            self.calls += 1
            return (self.calls - 1) % 2

        def observe(self, level, tokens, nbytes):
            self.seen.append((level, tokens, nbytes))

    pol = Alternate()
    sc = StreamingCodec(w.L, T, w.C, w.bins_k, w.bins_v, chunk_tokens=Tc, piece_chunks=1, fmt=fmt, levels=levels)
    pieces, outs, done = sc.roundtrip(torch.from_numpy(k).pin_memory(), torch.from_numpy(v).pin_memory(),
                                      policy=pol)
    done.synchronize()
    assert sc.status() == 0
    assert [hp.level for hp in pieces] == [0, 1, 0, 1]
    assert [lv for lv, _, _ in pol.seen] == [0, 1, 0, 1]
    for (ok, ov), hp in zip(outs, pieces):
        bk, bv = levels[hp.level]
        ks, vs = k[:, hp.t0:hp.t1].copy(), v[:, hp.t0:hp.t1].copy()
        if fmt == 2:
            ref = oracle_mod.compress_v2(ks, vs, Tc, bk, bv)
            rk, rv = oracle_mod.decompress_v2(ref["packed"], ref["off"], ref["len"], ref["rec"], ref["max1"], w.L,
                                              hp.t1 - hp.t0, w.C, Tc, bk, bv)
        else:
            ref = oracle_mod.compress_v3(ks, vs, Tc, bk, bv)
            rk, rv = oracle_mod.decompress_v3(ref["packed"], ref["len"], ref["side"], ref["max1"], w.L,
                                              hp.t1 - hp.t0, w.C, Tc, bk, bv)
        assert hp.nbytes == ref["packed"].size
        assert np.array_equal(hp.packed[:hp.nbytes].numpy(), ref["packed"])
        assert np.array_equal(ok.cpu().numpy().view(np.uint32), rk.view(np.uint32))
        assert np.array_equal(ov.cpu().numpy().view(np.uint32), rv.view(np.uint32))
