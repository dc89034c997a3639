"""Decompression straight into serving layouts ([CG §3.2]): binary16 output
equal to the oracle's rounding of the binary32 dequantisation, binary32 output
equal to cg_decompress_chunk's, both into [L, 2, T, C] caches, in both formats,
and untouched gaps between the layers' K and V planes."""
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


def _oracle_half(oracle_mod, k, v, bk, bv):
    """The coder is lossless, so the decoded symbols are the quantised ones."""
    sym, max1 = oracle_mod.quantize(k, v, bk, bv)
    return oracle_mod.dequantize_half(sym, max1, bk, bv)


@pytest.mark.parametrize("name,fmt", [("tiny", 1), ("tiny", 2), ("mistral_chunk", 1), ("mistral_chunk", 2)])
def test_half_into_paged_layout(cg, oracle_mod, synth_mod, name, fmt):
    w = synth_mod.WORKLOADS[name]
    k, v = synth_mod.generate(w)
    L, T, C_ = k.shape
    cd = cg.Codec(L, T, C_, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens, fmt=fmt)
    cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    cache = torch.full((L, 2, T + 3, C_), 7.0, dtype=torch.float16, device="cuda")  # gaps between planes
    cd.decompress_into(cache[:, 0, :T], cache[:, 1, :T])
    torch.cuda.synchronize()
    assert int(cd.dstatus.item()) == 0
    hk, hv = _oracle_half(oracle_mod, k, v, w.bins_k, w.bins_v)
    got = cache.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[:, 0, :T], hk)
    assert np.array_equal(got[:, 1, :T], hv)
    assert (cache[:, :, T:] == 7.0).all(), "rows outside the outputs were written"


@pytest.mark.parametrize("fmt", [1, 2])
def test_f32_into_paged_layout_equals_plain(cg, synth_mod, fmt):
    w = synth_mod.WORKLOADS["mistral_chunk"]
    k, v = synth_mod.generate(w, T=200)
    L, T, C_ = k.shape
    cd = cg.Codec(L, T, C_, w.bins_k, w.bins_v, chunk_tokens=64, fmt=fmt)
    cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    rk, rv = cd.decompress()
    rk, rv = rk.clone(), rv.clone()
    cache = torch.zeros((L, 2, T, C_), dtype=torch.float32, device="cuda")
    cd.decompress_into(cache[:, 0], cache[:, 1])
    torch.cuda.synchronize()
    assert torch.equal(cache[:, 0].view(torch.int32), rk.view(torch.int32))
    assert torch.equal(cache[:, 1].view(torch.int32), rv.view(torch.int32))


def test_half_odd_channels_generic_path(cg, oracle_mod):
    """C not a multiple of 4 takes the per-element writer."""
    rng = np.random.default_rng(4)
    L, T, C_, Tc = 2, 70, 6, 32
    k = rng.standard_normal((L, T, C_)).astype(np.float16)
    v = (rng.standard_normal((L, T, C_)) * 1e-3).astype(np.float16)
    bk, bv = [16, 7], [32, 4]
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc)
    cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    ok = torch.empty((L, T, C_), dtype=torch.float16, device="cuda")
    ov = torch.empty_like(ok)
    cd.decompress_into(ok, ov)
    torch.cuda.synchronize()
    hk, hv = _oracle_half(oracle_mod, k, v, bk, bv)
    assert np.array_equal(ok.cpu().numpy().view(np.uint16), hk)
    assert np.array_equal(ov.cpu().numpy().view(np.uint16), hv)
