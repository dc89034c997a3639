"""GPU parity: the CUDA library against the CPU oracle on the same seeded
inputs, through the C ABI. Integer outputs (symbols, max1 bits, CDF entries,
stream lengths, offsets, packed bytes) must match bit for bit; dequantised
binary32 output must be within 1e-6 relative (the same binary32 operations
run on both sides, so it is in fact checked bit for bit as well)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

REL_TOL = 1e-6


@pytest.fixture(scope="module")
def cg():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from kv_cache_compression_cg_gb300 import build, codec
    build.build()
    return codec


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def u16(t):
    return t.cpu().numpy().view(np.uint16)


def u32(t):
    return t.cpu().numpy().view(np.uint32)


def u64(t):
    return t.cpu().numpy().view(np.uint64)


def assert_close_f32(got, ref):
    got = np.asarray(got, np.float32)
    ref = np.asarray(ref, np.float32)
    scale = np.maximum(np.abs(ref), np.float32(1e-30))
    rel = np.abs(got.astype(np.float64) - ref.astype(np.float64)) / scale
    assert rel.max() <= REL_TOL, f"max rel err {rel.max()}"
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
        f"{int((got.view(np.uint32) != ref.view(np.uint32)).sum())} values differ in the last bits"


def _ragged(seed=42):
    rng = np.random.default_rng(seed)
    L, T, C_, Tc = 3, 150, 40, 64
    k = (rng.standard_normal((L, T, C_)) * rng.lognormal(0, 0.5, size=(1, 1, C_))).astype(np.float16)
    v = rng.standard_t(3, size=(L, T, C_)).astype(np.float16)
    k[1, 5] = 0.0
    v[2, 7] = -0.0
    k[0, 9, 3] = -70.0  # a negative group maximum
    return k, v, Tc, [32, 16, 8], [4, 16, 255]


def _shape_case(L, T, C_, Tc, bk, bv, seed):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((L, T, C_)) * 3).astype(np.float16)
    v = rng.uniform(-1, 1, size=(L, T, C_)).astype(np.float16)
    return k, v, Tc, bk, bv


def _synth(synth_mod, name, T=None):
    w = synth_mod.WORKLOADS[name]
    k, v = synth_mod.generate(w, T=T)
    return k, v, w.chunk_tokens, list(w.bins_k), list(w.bins_v)


CASES = ["tiny", "ragged", "c48_tc32_bins256", "c24_tc70", "c8_t1", "c16_tc1", "mistral_chunk",
         "uniform", "c24_tc600_bins255", "c136_bins64", "c40_bins20", "c64_bins24_36"]


def make_case(name, synth_mod):
    if name in ("tiny", "mistral_chunk", "uniform"):
        return _synth(synth_mod, name)
    if name == "ragged":
        return _ragged()
    if name == "c48_tc32_bins256":
        return _shape_case(2, 100, 48, 32, [256, 4], [8, 255], 1)
    if name == "c24_tc70":
        return _shape_case(2, 70, 24, 70, [16, 32], [32, 16], 2)
    if name == "c8_t1":
        return _shape_case(3, 1, 8, 256, [16, 16, 16], [4, 4, 4], 3)
    if name == "c16_tc1":
        return _shape_case(1, 5, 16, 1, [32], [32], 4)
    if name == "c24_tc600_bins255":  # chunks longer than 256 tokens (600, 600, then a ragged 100)
        return _shape_case(2, 1300, 24, 600, [255, 16], [32, 8], 5)
    if name == "c136_bins64":  # alphabets 33 .. 64: the fused kernel's 64-symbol form (a ragged last chunk)
        return _shape_case(3, 300, 136, 256, [64, 40, 16], [33, 64, 8], 6)
    if name == "c40_bins20":  # format-1 alphabets of 20 (not a multiple of 8): CDF entries stored one
        # by one; 176 slices, so the throughput kernel (the canary test runs a latency-mode size)
        return _shape_case(8, 1300, 40, 128, [20, 12] * 4, [12, 20] * 4, 7)
    if name == "c64_bins24_36":  # K rows of 24 entries (16-byte stores), V rows of 36 in the 64-symbol form
        return _shape_case(2, 260, 64, 256, [24, 16], [36, 10], 8)
    raise KeyError(name)


@pytest.mark.parametrize("case", CASES)
def test_compress_decompress_parity(cg, oracle_mod, synth_mod, case):
    k, v, Tc, bk, bv = make_case(case, synth_mod)
    L, T, C_ = k.shape
    ref = oracle_mod.compress(k, v, Tc, bk, bv)
    codec = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc)
    out = codec.compress(dev(k), dev(v))
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0
    assert np.array_equal(u16(out.max1), ref["max1"])
    assert np.array_equal(u16(out.cdf)[:ref["cdf"].size], ref["cdf"])
    assert np.array_equal(u32(out.len)[:ref["len"].size], ref["len"])
    assert np.array_equal(u64(out.off), ref["off"])
    total = int(ref["off"][-1])
    assert np.array_equal(out.packed[:total].cpu().numpy(), ref["packed"])
    ok, ov = codec.decompress()
    torch.cuda.synchronize()
    assert int(codec.dstatus.item()) == 0
    rk, rv = oracle_mod.decompress(ref["packed"], ref["off"], ref["len"], ref["cdf"], ref["max1"],
                                   L, T, C_, Tc, bk, bv)
    assert_close_f32(ok.cpu().numpy(), rk)
    assert_close_f32(ov.cpu().numpy(), rv)


@pytest.mark.parametrize("case", ["tiny", "ragged", "c48_tc32_bins256", "c24_tc70", "mistral_chunk",
                                  "c24_tc600_bins255"])
def test_step_functions_parity(cg, oracle_mod, synth_mod, case):
    k, v, Tc, bk, bv = make_case(case, synth_mod)
    L, T, C_ = k.shape
    A_k, A_v = max(bk), max(bv)
    sym_ref, max1_ref = oracle_mod.quantize(k, v, bk, bv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sym, max1 = cg.quantize(dev(k), dev(v), bk, bv, chunk_tokens=Tc, status=status)
    assert np.array_equal(sym.cpu().numpy(), sym_ref)
    assert np.array_equal(u16(max1), max1_ref)
    cdf_ref = oracle_mod.calculate_cdf(sym_ref, Tc, A_k, A_v)
    cdf = cg.calculate_cdf(sym, bk, bv, chunk_tokens=Tc, status=status)
    assert np.array_equal(u16(cdf)[:cdf_ref.size], cdf_ref)
    packed_ref, len_ref, off_ref, st = oracle_mod.encode(sym_ref, cdf_ref, Tc, A_k, A_v)
    assert st == 0
    packed, ln, off = cg.encode(sym, cdf, bk, bv, chunk_tokens=Tc, status=status)
    assert np.array_equal(u32(ln)[:len_ref.size], len_ref)
    assert np.array_equal(u64(off), off_ref)
    assert np.array_equal(packed[:int(off_ref[-1])].cpu().numpy(), packed_ref)
    sym2 = cg.decode(packed, off, ln, cdf, L, T, C_, bk, bv, chunk_tokens=Tc, status=status)
    assert np.array_equal(sym2.cpu().numpy(), sym_ref)
    ok, ov = cg.dequantize(sym2, max1, bk, bv, chunk_tokens=Tc)
    rk, rv = oracle_mod.dequantize(sym_ref, max1_ref, bk, bv)
    assert_close_f32(ok.cpu().numpy(), rk)
    assert_close_f32(ov.cpu().numpy(), rv)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_ctx4096_full_parity(cg, oracle_mod, synth_mod):
    """The 32 x 4096 x 1024 workload in 16 chunks, one batched call, every
    output compared with the oracle."""
    k, v, Tc, bk, bv = _synth(synth_mod, "ctx4096")
    L, T, C_ = k.shape
    ref = oracle_mod.compress(k, v, Tc, bk, bv)
    codec = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc)
    out = codec.compress(dev(k), dev(v))
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0
    assert np.array_equal(u16(out.max1), ref["max1"])
    assert np.array_equal(u16(out.cdf), ref["cdf"])
    assert np.array_equal(u32(out.len), ref["len"])
    assert np.array_equal(u64(out.off), ref["off"])
    total = int(ref["off"][-1])
    assert np.array_equal(out.packed[:total].cpu().numpy(), ref["packed"])
    ok, ov = codec.decompress()
    torch.cuda.synchronize()
    assert int(codec.dstatus.item()) == 0
    rk, rv = oracle_mod.decompress(ref["packed"], ref["off"], ref["len"], ref["cdf"], ref["max1"],
                                   L, T, C_, Tc, bk, bv)
    assert_close_f32(ok.cpu().numpy(), rk)
    assert_close_f32(ov.cpu().numpy(), rv)


def test_vllm_layout_views(cg, oracle_mod):
    """K and V as views of one [L, 2, T, C] tensor (layer stride 2*T*C)."""
    rng = np.random.default_rng(8)
    L, T, C_ = 4, 96, 64
    kv = (rng.standard_normal((L, 2, T, C_)) * 2).astype(np.float16)
    bk = [32, 32, 16, 16]
    t = dev(kv)
    codec = cg.Codec(L, T, C_, bk, chunk_tokens=32)
    out = codec.compress(t[:, 0], t[:, 1])
    torch.cuda.synchronize()
    ref = oracle_mod.compress(kv[:, 0].copy(), kv[:, 1].copy(), 32, bk, bk)
    assert np.array_equal(u64(out.off), ref["off"])
    assert np.array_equal(out.packed[:int(ref["off"][-1])].cpu().numpy(), ref["packed"])
    assert np.array_equal(u16(out.cdf), ref["cdf"])


def test_nonfinite_input_flagged(cg):
    k = torch.randn(2, 64, 64, device="cuda").half()
    v = torch.randn(2, 64, 64, device="cuda").half()
    k[1, 3, 5] = float("inf")
    codec = cg.Codec(2, 64, 64, [16, 16], chunk_tokens=64)
    out = codec.compress(k, v)
    torch.cuda.synchronize()
    assert int(out.status.item()) & 0x1


def test_capacity_shortfall(cg, oracle_mod, synth_mod):
    k, v, Tc, bk, bv = make_case("tiny", synth_mod)
    L, T, C_ = k.shape
    ref = oracle_mod.compress(k, v, Tc, bk, bv)
    cap = int(ref["off"][-1]) // 2 + 3
    codec = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, capacity=cap)
    codec.out.packed.fill_(0xAB)
    out = codec.compress(dev(k), dev(v))
    torch.cuda.synchronize()
    assert int(out.status.item()) & 0x2
    assert np.array_equal(u64(out.off), ref["off"])
    got = out.packed.cpu().numpy()
    assert np.array_equal(got[:cap], ref["packed"][:cap])
    assert (got[cap:] == 0xAB).all(), "bytes past the capacity were written"


def test_corrupted_stream_matches_oracle_and_flags(cg, oracle_mod, synth_mod):
    k, v, Tc, bk, bv = make_case("ragged", synth_mod)
    L, T, C_ = k.shape
    ref = oracle_mod.compress(k, v, Tc, bk, bv)
    bad = ref["packed"].copy()
    rng = np.random.default_rng(0)
    idx = rng.integers(0, bad.size, size=40)
    bad[idx] ^= 0x5A
    sym_ref, st_ref = oracle_mod.decode(bad, ref["off"], ref["len"], ref["cdf"], L, T, C_, Tc,
                                        max(bk), max(bv))
    assert st_ref == oracle_mod.ERR_CORRUPT
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    padded = np.zeros(bad.size + 16, np.uint8)
    padded[:bad.size] = bad
    sym = cg.decode(dev(padded), dev(ref["off"].view(np.int64)), dev(ref["len"].view(np.int32)),
                    dev(ref["cdf"].view(np.int16)), L, T, C_, bk, bv, chunk_tokens=Tc,
                    status=status, packed_bytes=bad.size)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x4
    assert np.array_equal(sym.cpu().numpy(), sym_ref)


def test_offsets_outside_buffer_flagged(cg, oracle_mod, synth_mod):
    k, v, Tc, bk, bv = make_case("tiny", synth_mod)
    L, T, C_ = k.shape
    ref = oracle_mod.compress(k, v, Tc, bk, bv)
    off = ref["off"].copy()
    off[5] = np.uint64(1 << 40)  # far outside the buffer
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cg.decode(dev(np.append(ref["packed"], np.zeros(16, np.uint8))), dev(off.view(np.int64)),
              dev(ref["len"].view(np.int32)), dev(ref["cdf"].view(np.int16)), L, T, C_, bk, bv,
              chunk_tokens=Tc, status=status, packed_bytes=ref["packed"].size)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x4


def test_bad_symbol_flagged(cg, oracle_mod):
    rng = np.random.default_rng(1)
    sym = rng.integers(0, 16, size=(2, 2, 64, 32)).astype(np.uint8)
    cdf = oracle_mod.calculate_cdf(sym, 64, 16, 16)
    sym[1, 0, 3, 4] = 200
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cg.encode(dev(sym), dev(cdf.view(np.int16)), [16, 16], [16, 16], chunk_tokens=64, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x8


def test_empty_token_range(cg):
    k = torch.empty((2, 0, 64), dtype=torch.float16, device="cuda")
    codec = cg.Codec(2, 0, 64, [16, 16], chunk_tokens=64)
    codec.out.off.fill_(-1)
    out = codec.compress(k, k)
    torch.cuda.synchronize()
    assert out.off.cpu().tolist() == [0]
