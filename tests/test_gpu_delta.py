"""GPU parity for the token-locality delta (the change-based encoding of
[CG §1.2(1)]): the step kernels (quantise, dequantise) and the fused
compress / decompress in both formats against the oracle on the same seeded
inputs, bit for bit, across group sizes that divide the chunk, do not, and
exceed it, ragged chunks, the vector and the generic kernels, binary16 output
into a [L, 2, T, C] cache, and non-finite input flagged."""
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


def _correlated(seed, L, T, C_, rho=0.97):
    rng = np.random.default_rng(seed)
    off = rng.standard_normal((L, 1, C_)) * rng.lognormal(0, 0.7, (1, 1, C_))
    x = np.empty((L, T, C_))
    x[:, 0] = rng.standard_normal((L, C_))
    for t in range(1, T):
        x[:, t] = rho * x[:, t - 1] + np.sqrt(1 - rho * rho) * rng.standard_normal((L, C_))
    return (x * 0.5 + off).astype(np.float16)


# (L, T, C, Tc, bins_k, bins_v, group): vector kernels (C % 8 == 0), the generic
# kernel (C = 6, C = 4096), groups dividing the chunk, not dividing it, larger
# than it, ragged last chunks
STEP_CASES = {
    "g2": (2, 100, 64, 32, [16, 8], [32, 4], 2),
    "g10_ragged": (3, 300, 40, 64, [32, 16, 8], [16, 16, 16], 10),
    "g7_c1024": (2, 70, 1024, 64, [16, 32], [32, 16], 7),
    "g300": (1, 130, 32, 64, [16], [16], 300),
    "odd_c": (2, 50, 6, 16, [8, 256], [5, 33], 3),
    "wide_c": (1, 20, 4096, 16, [16], [8], 4),
}


@pytest.mark.parametrize("case", list(STEP_CASES))
def test_quantize_dequantize_delta_steps(cg, oracle_mod, case):
    L, T, C_, Tc, bk, bv, G = STEP_CASES[case]
    k = _correlated(1, L, T, C_)
    v = _correlated(2, L, T, C_, rho=0.8)
    sym, max1 = cg.quantize_delta(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), G, bk, bv,
                                  chunk_tokens=Tc)
    rs, rm = oracle_mod.quantize_delta(k, v, Tc, G, bk, bv)
    assert np.array_equal(max1.cpu().numpy().view(np.uint16), rm)
    assert np.array_equal(sym.cpu().numpy(), rs)
    ok, ov = cg.dequantize_delta(sym, max1, G, bk, bv, chunk_tokens=Tc)
    wk, wv = oracle_mod.dequantize_delta(rs, rm, Tc, G, bk, bv)
    torch.cuda.synchronize()
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), wv.view(np.uint32))


FUSED_CASES = {
    "g10": (2, 200, 64, 64, [32, 16], [16, 8], 10),
    "g4_ragged": (3, 300, 40, 128, [16, 32, 8], [8, 16, 32], 4),
    "g3_tc256": (2, 520, 128, 256, [16, 16], [32, 32], 3),
    "g256": (1, 256, 64, 256, [32], [16], 256),
    "g2_t1": (2, 1, 16, 64, [16, 8], [8, 16], 2),
    "g10_bins64": (2, 300, 136, 256, [64, 34], [48, 16], 10),  # the fused kernel's 64-symbol form
}


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("case", list(FUSED_CASES))
def test_fused_delta_matches_oracle(cg, oracle_mod, case, fmt):
    L, T, C_, Tc, bk, bv, G = FUSED_CASES[case]
    k = _correlated(3, L, T, C_)
    v = _correlated(4, L, T, C_, rho=0.9)
    ref = oracle_mod.compress_ex(k, v, Tc, bk, bv, fmt=fmt, group=G)
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=fmt, group=G)
    out = cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    ok, ov = cd.decompress()
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0 and int(cd.dstatus.item()) == 0
    assert np.array_equal(out.max1.cpu().numpy().view(np.uint16), ref["max1"])
    if fmt == 1:
        assert np.array_equal(out.cdf[:cd.cdf_elems].cpu().numpy().view(np.uint16), ref["cdf"])
    else:
        assert np.array_equal(out.rec[:cd.rec_bytes].cpu().numpy(), ref["rec"])
    ns = 2 * L * T
    assert np.array_equal(out.len[:ns].cpu().numpy().view(np.uint32), ref["len"])
    assert np.array_equal(out.off.cpu().numpy().view(np.uint64), ref["off"])
    total = int(ref["off"][-1])
    assert np.array_equal(out.packed[:total].cpu().numpy(), ref["packed"])
    side = ref["cdf"] if fmt == 1 else ref["rec"]
    wk, wv = oracle_mod.decompress_ex(ref["packed"], ref["off"], ref["len"], side, ref["max1"], L, T, C_, Tc,
                                      bk, bv, fmt=fmt, group=G)
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), wv.view(np.uint32))
    # binary16 straight into a [L, 2, T, C] cache
    cache = torch.zeros((L, 2, T, C_), dtype=torch.float16, device="cuda")
    cd.decompress_into(cache[:, 0], cache[:, 1])
    torch.cuda.synchronize()
    got = cache.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[:, 0], oracle_mod.floats_to_half(wk))
    assert np.array_equal(got[:, 1], oracle_mod.floats_to_half(wv))


@pytest.mark.parametrize("fmt", [1, 2, 3])
def test_generic_compress_path_with_delta(cg, oracle_mod, fmt):
    """C % 8 != 0 takes the step kernels (quantise with the delta, slice
    coder, scan) inside the compress entry points, in every format (format 2
    with a 64-bin layer, whose alphabet is past the fused kernel's too); the
    decoder stays fused."""
    L, T, C_, Tc, G = 2, 150, 12, 64, 5
    bk, bv = ([16, 32], [8, 16]) if fmt == 3 else ([16, 64], [8, 16])
    k = _correlated(5, L, T, C_)
    v = _correlated(6, L, T, C_)
    if fmt == 3:
        ref = oracle_mod.compress_v3(k, v, Tc, bk, bv, group=G)
    else:
        ref = oracle_mod.compress_ex(k, v, Tc, bk, bv, fmt=fmt, group=G)
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=fmt, group=G)
    out = cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    ok, ov = cd.decompress()
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0 and int(cd.dstatus.item()) == 0
    assert np.array_equal(out.max1.cpu().numpy().view(np.uint16), ref["max1"])
    assert np.array_equal(out.len[:2 * L * T].cpu().numpy().view(np.uint32), ref["len"])
    assert np.array_equal(out.off.cpu().numpy().view(np.uint64), ref["off"])
    assert np.array_equal(out.packed[:int(ref["off"][-1])].cpu().numpy(), ref["packed"])
    if fmt == 1:
        assert np.array_equal(out.cdf[:cd.cdf_elems].cpu().numpy().view(np.uint16), ref["cdf"])
        wk, wv = oracle_mod.decompress_ex(ref["packed"], ref["off"], ref["len"], ref["cdf"], ref["max1"],
                                          L, T, C_, Tc, bk, bv, fmt=1, group=G)
    elif fmt == 2:
        assert np.array_equal(out.rec[:cd.rec_bytes].cpu().numpy(), ref["rec"])
        wk, wv = oracle_mod.decompress_ex(ref["packed"], ref["off"], ref["len"], ref["rec"], ref["max1"],
                                          L, T, C_, Tc, bk, bv, fmt=2, group=G)
    else:
        assert np.array_equal(out.side3[:out.side3_bytes()].cpu().numpy(), ref["side"])
        wk, wv = oracle_mod.decompress_v3(ref["packed"], ref["len"], ref["side"], ref["max1"],
                                          L, T, C_, Tc, bk, bv, group=G)
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), wv.view(np.uint32))


def test_delta_lowers_error_on_synthetic_cache(cg, synth_mod):
    """On the seeded stand-in for a model's KV cache (AR(1) tokens), the delta
    reconstructs with less error than plain quantisation at the same bins."""
    w = synth_mod.WORKLOADS["mistral_chunk"]
    k, v = synth_mod.generate(w)
    L, T, C_ = k.shape
    kt, vt = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    errs = []
    for G in (1, 4):
        cd = cg.Codec(L, T, C_, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens, fmt=2, group=G)
        cd.compress(kt, vt)
        ok, _ = cd.decompress()
        errs.append(float(((ok - kt.float()) ** 2).mean().sqrt()))
    assert errs[1] < errs[0]


def test_nonfinite_flagged_with_delta(cg):
    L, T, C_ = 1, 64, 64
    k = torch.zeros((L, T, C_), dtype=torch.float16, device="cuda")
    k[0, 5, 7] = float("inf")  # a delta row of group 0 (G = 4)
    v = torch.zeros_like(k)
    for fmt in (1, 2):
        cd = cg.Codec(L, T, C_, [16], [16], chunk_tokens=64, fmt=fmt, group=4)
        out = cd.compress(k, v)
        torch.cuda.synchronize()
        assert int(out.status.item()) & 1


@pytest.mark.slow
def test_fused_delta_full_workload(cg, oracle_mod, synth_mod):
    """The benchmark's 4096-token workload with groups of 10, format 2, in
    the launch configuration `bench.py --group 10` times: every output equal
    to the oracle's."""
    w = synth_mod.WORKLOADS["ctx4096"]
    k, v = synth_mod.generate(w)
    L, T, C_, Tc, G = w.L, w.T, w.C, w.chunk_tokens, 10
    ref = oracle_mod.compress_ex(k, v, Tc, w.bins_k, w.bins_v, fmt=2, group=G)
    cd = cg.Codec(L, T, C_, w.bins_k, w.bins_v, chunk_tokens=Tc, fmt=2, group=G)
    out = cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    ok, ov = cd.decompress()
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0 and int(cd.dstatus.item()) == 0
    assert np.array_equal(out.max1.cpu().numpy().view(np.uint16), ref["max1"])
    assert np.array_equal(out.rec[:cd.rec_bytes].cpu().numpy(), ref["rec"])
    assert np.array_equal(out.off.cpu().numpy().view(np.uint64), ref["off"])
    assert np.array_equal(out.packed[:int(ref["off"][-1])].cpu().numpy(), ref["packed"])
    wk, wv = oracle_mod.decompress_ex(ref["packed"], ref["off"], ref["len"], ref["rec"], ref["max1"], L, T, C_,
                                      Tc, w.bins_k, w.bins_v, fmt=2, group=G)
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), wv.view(np.uint32))


def test_long_chunks_decode_through_the_steps(cg, oracle_mod):
    """Chunks over 256 tokens: cg_compress_chunk_ex (format 1) takes the step
    kernels, and the symbols decode with cg_decode then cg_dequantize_delta;
    both equal the oracle's."""
    from kv_cache_compression_cg_gb300 import capi
    import ctypes as C
    L, T, C_, Tc, G = 2, 700, 32, 512, 10
    bk, bv = [16, 32], [8, 16]
    k = _correlated(7, L, T, C_)
    v = _correlated(8, L, T, C_)
    ref = oracle_mod.compress_ex(k, v, Tc, bk, bv, fmt=1, group=G)
    lib = capi.load()
    shp = cg.make_shape(L, T, C_, Tc)
    bka, bva = np.array(bk, np.int32), np.array(bv, np.int32)
    n_cdf = int(lib.cg_cdf_elems(C.byref(shp), bka.ctypes.data, bva.ctypes.data))
    cap = int(lib.cg_max_compressed_bytes(C.byref(shp)))
    ws_n = int(lib.cg_compress_workspace_bytes(C.byref(shp)))
    dev = "cuda"
    kt, vt = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    max1 = torch.empty((2, L, T), dtype=torch.int16, device=dev)
    cdf = torch.empty(n_cdf, dtype=torch.int16, device=dev)
    packed = torch.empty(cap, dtype=torch.uint8, device=dev)
    ln = torch.empty(2 * L * T, dtype=torch.int32, device=dev)
    off = torch.empty(2 * L * T + 1, dtype=torch.int64, device=dev)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    p = lambda t: C.c_void_p(t.data_ptr())
    s = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    capi.check(lib.cg_compress_chunk_ex(p(kt), p(vt), C.byref(shp), bka.ctypes.data, bva.ctypes.data, 1, G, p(max1),
                                        p(cdf), p(packed), cap, p(ln), p(off), p(ws), ws_n, p(st), s),
               "cg_compress_chunk_ex")
    sym = cg.decode(packed, off, ln, cdf, L, T, C_, bk, bv, chunk_tokens=Tc, status=st)
    ok, ov = cg.dequantize_delta(sym, max1, G, bk, bv, chunk_tokens=Tc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(max1.cpu().numpy().view(np.uint16), ref["max1"])
    assert np.array_equal(cdf.cpu().numpy().view(np.uint16), ref["cdf"])
    assert np.array_equal(packed[:int(ref["off"][-1])].cpu().numpy(), ref["packed"])
    wk, wv = oracle_mod.decompress_ex(ref["packed"], ref["off"], ref["len"], ref["cdf"], ref["max1"], L, T, C_, Tc,
                                      bk, bv, fmt=1, group=G)
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), wv.view(np.uint32))
