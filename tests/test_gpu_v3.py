"""GPU parity for format 3 (compact count records): the side buffer, max1,
lengths, offsets and packed bytes equal the oracle's bit for bit, the streams
equal format 2's, decompression from the lengths alone gives the oracle's
values (binary32, and binary16 into a [L, 2, T, C] cache), with and without
the token-locality delta; malformed side buffers are flagged."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from kv_cache_compression_cg_gb300 import build, codec
    build.build()
    return codec


def _case(synth_mod, name):
    if name in ("tiny", "mistral_chunk", "ctx4096"):
        w = synth_mod.WORKLOADS[name]
        k, v = synth_mod.generate(w)
        return k, v, w.chunk_tokens, list(w.bins_k), list(w.bins_v)
    rng = np.random.default_rng(len(name) + 50)
    shapes = {"ragged": (3, 200, 40, 64, [32, 16, 8], [16, 16, 16]),
              "odd_bins": (2, 96, 16, 32, [7, 5], [33, 4]),
              "t1": (2, 1, 8, 256, [16, 32], [4, 8]),
              "odd_c": (2, 70, 13, 64, [16, 32], [8, 33])}  # C % 8 != 0: the step path
    L, T, C_, Tc, bk, bv = shapes[name]
    k = (rng.standard_normal((L, T, C_)) * rng.lognormal(0, 0.5, (1, 1, C_))).astype(np.float16)
    v = (rng.standard_normal((L, T, C_)) * 0.5).astype(np.float16)
    return k, v, Tc, bk, bv


@pytest.mark.parametrize("G", [1, 10])
@pytest.mark.parametrize("case", ["tiny", "ragged", "odd_bins", "t1", "odd_c", "mistral_chunk",
                                  pytest.param("ctx4096", marks=pytest.mark.slow)])
def test_v3_parity_with_oracle(cg, oracle_mod, synth_mod, case, G):
    k, v, Tc, bk, bv = _case(synth_mod, case)
    L, T, C_ = k.shape
    ref = oracle_mod.compress_v3(k, v, Tc, bk, bv, group=G)
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=3, group=G)
    out = cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    ok, ov = cd.decompress()
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0 and int(cd.dstatus.item()) == 0
    n = out.side3_bytes()
    assert n == ref["side"].size
    assert np.array_equal(out.side3[:n].cpu().numpy(), ref["side"])
    assert np.array_equal(out.max1.cpu().numpy().view(np.uint16), ref["max1"])
    ns = 2 * L * T
    assert np.array_equal(out.len[:ns].cpu().numpy().view(np.uint32), ref["len"])
    assert np.array_equal(out.off.cpu().numpy().view(np.uint64), ref["off"])
    assert np.array_equal(out.packed[:int(ref["off"][-1])].cpu().numpy(), ref["packed"])
    wk, wv = oracle_mod.decompress_v3(ref["packed"], ref["len"], ref["side"], ref["max1"], L, T, C_, Tc, bk, bv,
                                      group=G)
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), wv.view(np.uint32))
    # binary16 straight into a [L, 2, T, C] cache
    cache = torch.zeros((L, 2, T, C_), dtype=torch.float16, device="cuda")
    cd.decompress_into(cache[:, 0], cache[:, 1])
    torch.cuda.synchronize()
    got = cache.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[:, 0], oracle_mod.floats_to_half(wk))
    assert np.array_equal(got[:, 1], oracle_mod.floats_to_half(wv))


def test_v3_streams_equal_v2_and_side_is_smaller(cg, synth_mod):
    w = synth_mod.WORKLOADS["mistral_chunk"]
    k, v = synth_mod.generate(w)
    kt, vt = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    c2 = cg.Codec(w.L, w.T, w.C, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens, fmt=2)
    c3 = cg.Codec(w.L, w.T, w.C, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens, fmt=3)
    o2, o3 = c2.compress(kt, vt), c3.compress(kt, vt)
    torch.cuda.synchronize()
    total = int(o2.off[-1].item())
    assert torch.equal(o2.packed[:total], o3.packed[:total])
    assert torch.equal(o2.len, o3.len) and torch.equal(o2.off, o3.off)
    assert o3.side3_bytes() < 0.5 * c2.rec_bytes


def test_v3_malformed_side_flagged(cg, synth_mod, oracle_mod):
    """Each corruption sets CG_FLAG_CORRUPT and the decoder stays in bounds."""
    k, v, Tc, bk, bv = _case(synth_mod, "ragged")
    L, T, C_ = k.shape
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=3)
    out = cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    torch.cuda.synchronize()
    good = out.side3.clone()
    nch = -(-T // Tc)
    ns = 2 * L * nch
    offM = 8 * (ns + 1)
    offB = (offM + ns * C_ + 3) // 4 * 4

    def run(mutate):
        out.side3.copy_(good)
        mutate(out.side3)
        cd.dstatus.zero_()
        cd.decompress()
        torch.cuda.synchronize()
        return int(cd.dstatus.item())

    assert run(lambda s: None) == 0
    assert run(lambda s: s.__setitem__(offM, 200)) & 4                     # mode outside the alphabet
    assert run(lambda s: s[offB:offB + 4].copy_(torch.tensor([255, 255, 255, 255], dtype=torch.uint8))) & 4
    assert run(lambda s: s[8:16].copy_(torch.tensor([255] * 8, dtype=torch.uint8))) & 4  # O[1] out of range
    assert run(lambda s: s[8 * ns:8 * ns + 8].copy_(torch.tensor([255] * 8, dtype=torch.uint8))) & 4  # |V|


def test_v3_streaming(cg, synth_mod, oracle_mod):
    from kv_cache_compression_cg_gb300.stream import StreamingCodec
    w = synth_mod.WORKLOADS["mistral_chunk"]
    T, Tc = 200, 64
    k, v = synth_mod.generate(w, T=T)
    sc = StreamingCodec(w.L, T, w.C, w.bins_k, w.bins_v, chunk_tokens=Tc, piece_chunks=2, fmt=3)
    pieces, outs, done = sc.roundtrip(torch.from_numpy(k).pin_memory(), torch.from_numpy(v).pin_memory())
    done.synchronize()
    assert sc.status() == 0
    rk, rv = oracle_mod.decompress_v3(*[oracle_mod.compress_v3(k, v, Tc, w.bins_k, w.bins_v)[key]
                                        for key in ("packed", "len", "side", "max1")], w.L, T, w.C, Tc,
                                      w.bins_k, w.bins_v)
    for (ok, ov), hp in zip(outs, pieces):
        assert np.array_equal(ok.cpu().numpy().view(np.uint32), rk[:, hp.t0:hp.t1].view(np.uint32))
        assert np.array_equal(ov.cpu().numpy().view(np.uint32), rv[:, hp.t0:hp.t1].view(np.uint32))
