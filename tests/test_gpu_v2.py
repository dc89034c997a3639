"""GPU parity for format 2 (count records instead of CDF entries): the CUDA
library against the oracle's format 2 on the same seeded inputs, bit for bit
(max1, records, lengths, offsets, packed bytes, dequantised binary32), format
2 decoding to exactly format 1's values, corrupt records flagged, and the
streaming path in format 2."""
import numpy as np
import pytest
import torch

from kv_cache_compression_cg_gb300 import shard

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from kv_cache_compression_cg_gb300 import build, codec
    build.build()
    return codec


def _case(synth_mod, name):
    if name in ("tiny", "mistral_chunk", "uniform", "ctx4096"):
        w = synth_mod.WORKLOADS[name]
        k, v = synth_mod.generate(w)
        return k, v, w.chunk_tokens, list(w.bins_k), list(w.bins_v)
    rng = np.random.default_rng(len(name))
    shapes = {"ragged": (3, 200, 40, 64, [32, 16, 8], [16, 16, 16]),
              "odd_bins": (2, 96, 16, 32, [7, 5], [33, 4]),
              "t1": (2, 1, 8, 256, [16, 32], [4, 8]),
              "tc1": (1, 5, 16, 1, [32], [32]),
              # past the fused kernel: alphabets up to 255 symbols, C % 8 != 0
              "wide_bins": (3, 300, 40, 128, [256, 64, 255], [128, 34, 4]),
              "odd_c": (2, 70, 13, 64, [16, 32], [8, 4]),
              # the fused kernel's 64-symbol form: layer alphabets 33 .. 63 (bins up to 65)
              "bins65": (3, 300, 136, 256, [65, 48, 16], [34, 64, 8])}
    L, T, C_, Tc, bk, bv = shapes[name]
    k = (rng.standard_normal((L, T, C_)) * rng.lognormal(0, 0.5, (1, 1, C_))).astype(np.float16)
    v = (rng.standard_normal((L, T, C_)) * 0.5).astype(np.float16)
    return k, v, Tc, bk, bv


CASES = ["tiny", "ragged", "odd_bins", "t1", "tc1", "wide_bins", "odd_c", "bins65", "mistral_chunk", "uniform"]


@pytest.mark.parametrize("case", CASES + [pytest.param("ctx4096", marks=pytest.mark.slow)])
def test_v2_parity_with_oracle(cg, oracle_mod, synth_mod, case):
    k, v, Tc, bk, bv = _case(synth_mod, case)
    L, T, C_ = k.shape
    ref = oracle_mod.compress_v2(k, v, Tc, bk, bv)
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=2)
    out = cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    ok, ov = cd.decompress()
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0 and int(cd.dstatus.item()) == 0
    assert cd.rec_bytes == ref["rec"].size
    assert np.array_equal(out.max1.cpu().numpy().view(np.uint16), ref["max1"])
    assert np.array_equal(out.rec[:cd.rec_bytes].cpu().numpy(), ref["rec"])
    ns = 2 * L * T
    assert np.array_equal(out.len[:ns].cpu().numpy().view(np.uint32), ref["len"])
    assert np.array_equal(out.off.cpu().numpy().view(np.uint64), ref["off"])
    total = int(ref["off"][-1])
    assert np.array_equal(out.packed[:total].cpu().numpy(), ref["packed"])
    rk, rv = oracle_mod.decompress_v2(ref["packed"], ref["off"], ref["len"], ref["rec"], ref["max1"],
                                      L, T, C_, Tc, bk, bv)
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), rv.view(np.uint32))
    # format 1 of the same input decodes to the same values
    cd1 = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc)
    cd1.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    ok1, ov1 = cd1.decompress()
    torch.cuda.synchronize()
    assert torch.equal(ok.view(torch.int32), ok1.view(torch.int32))
    assert torch.equal(ov.view(torch.int32), ov1.view(torch.int32))
    # and its side information is smaller
    assert cd.rec_bytes < 2 * cd1.cdf_elems


def test_v2_corrupt_records_flagged(cg, oracle_mod, synth_mod):
    k, v, Tc, bk, bv = _case(synth_mod, "tiny")
    L, T, C_ = k.shape
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=2)
    out = cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    torch.cuda.synchronize()
    rec = out.rec.clone()
    A0 = oracle_mod.alphabet_v2(bk[0])
    out.rec[0] = A0 + 3                      # mode byte outside the alphabet
    out.rec[A0 + 1:2 * A0] = 255             # counts above the chunk's tokens
    cd.decompress()
    torch.cuda.synchronize()
    assert int(cd.dstatus.item()) & 0x4
    out.rec.copy_(rec)
    cd.dstatus.zero_()
    cd.decompress()
    torch.cuda.synchronize()
    assert int(cd.dstatus.item()) == 0


def test_v2_layer_views(cg, oracle_mod, synth_mod):
    """K and V as views of one [L, 2, T, C] tensor (layer stride 2*T*C)."""
    k, v, Tc, bk, bv = _case(synth_mod, "mistral_chunk")
    L, T, C_ = k.shape
    kv = torch.empty((L, 2, T, C_), dtype=torch.float16, device="cuda")
    kv[:, 0] = torch.from_numpy(k).cuda()
    kv[:, 1] = torch.from_numpy(v).cuda()
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=2)
    out = cd.compress(kv[:, 0], kv[:, 1])
    torch.cuda.synchronize()
    ref = oracle_mod.compress_v2(k, v, Tc, bk, bv)
    assert np.array_equal(out.rec[:cd.rec_bytes].cpu().numpy(), ref["rec"])
    assert np.array_equal(out.packed[:int(ref["off"][-1])].cpu().numpy(), ref["packed"])


def test_v2_stream_matches_oracle(cg, oracle_mod, synth_mod):
    from kv_cache_compression_cg_gb300.stream import StreamingCodec
    w = synth_mod.WORKLOADS["mistral_chunk"]
    T, Tc = 200, 32
    k, v = synth_mod.generate(w, T=T)
    sc = StreamingCodec(w.L, T, w.C, w.bins_k, w.bins_v, chunk_tokens=Tc, piece_chunks=2, fmt=2)
    pieces, outs, done = sc.roundtrip(torch.from_numpy(k).pin_memory(), torch.from_numpy(v).pin_memory())
    done.synchronize()
    assert sc.status() == 0
    joined = shard.assemble([hp.arrays() for hp in pieces])
    ref = oracle_mod.compress_v2(k, v, Tc, w.bins_k, w.bins_v)
    for key in ("max1", "rec", "packed", "len", "off"):
        assert np.array_equal(joined[key], ref[key]), key
    rk, rv = oracle_mod.decompress_v2(ref["packed"], ref["off"], ref["len"], ref["rec"], ref["max1"],
                                      w.L, T, w.C, Tc, w.bins_k, w.bins_v)
    for (ok, ov), hp in zip(outs, pieces):
        assert np.array_equal(ok.cpu().numpy().view(np.uint32), rk[:, hp.t0:hp.t1].view(np.uint32))
        assert np.array_equal(ov.cpu().numpy().view(np.uint32), rv[:, hp.t0:hp.t1].view(np.uint32))
