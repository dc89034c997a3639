"""Degenerate and extreme inputs through every side-information format, with
and without the token-locality delta, on the GPU against the oracle, bit for
bit (max1, side information, lengths, offsets, packed bytes, decoded values):

- an all-zero layer (max1 = 0: every symbol is MAX and one symbol takes the
  whole CDF but A - 1);
- constant rows (every symbol 2 MAX) and negative constant rows (every symbol 0);
- rows at the largest finite binary16, +-65504, mixed with subnormals and
  signed zeros (with the delta, max |d| exceeds 65504 and max1 saturates, so
  the clamp decides the symbols);
- rows of subnormals only (max1 subnormal, MAX / max1 large but finite);
- an all-zero token row and an all -0 token row inside random data;
- three chunks of 64, 64 and 22 tokens (a ragged last chunk), and delta groups
  that divide the chunk, do not, and exceed it."""
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


def _extremes(fmt):
    L, T, C_, Tc = 4, 150, 32, 64
    rng = np.random.default_rng(7)
    k = np.zeros((L, T, C_), np.float16)
    v = np.zeros((L, T, C_), np.float16)
    # layer 0: K all zero; V constant 1.0
    v[0] = 1.0
    # layer 1: K at +-65504 with subnormals and signed zeros; V subnormals only
    k[1] = rng.choice(np.array([65504.0, -65504.0, 0.0, -0.0, 2.0 ** -24, -(2.0 ** -24), 1.0]),
                      size=(T, C_)).astype(np.float16)
    v[1] = (rng.integers(-1023, 1024, size=(T, C_)) * 2.0 ** -24).astype(np.float16)
    # layer 2: K small values with one channel at 65504; V negative constant rows
    k[2] = (rng.standard_normal((T, C_)) * 1e-3).astype(np.float16)
    k[2, :, 0] = 65504.0
    v[2] = (-np.linspace(0.5, 100.0, T)[:, None] * np.ones((1, C_))).astype(np.float16)
    # layer 3: random, with an all-zero row and an all -0 row
    k[3] = rng.standard_normal((T, C_)).astype(np.float16)
    k[3, 10] = 0.0
    k[3, 11] = -0.0
    v[3] = rng.standard_t(3, size=(T, C_)).astype(np.float16)
    if fmt == 3:  # compact records: every layer alphabet within 32 symbols
        bk, bv = [32, 4, 32, 16], [16, 32, 8, 33]
    else:  # the widest alphabets take the step path
        bk, bv = [32, 4, 256, 16], [16, 32, 8, 255]
    return k, v, Tc, bk, bv


@pytest.mark.parametrize("G", [1, 4, 10, 100])
@pytest.mark.parametrize("fmt", [1, 2, 3])
def test_extremes_match_oracle(cg, oracle_mod, fmt, G):
    k, v, Tc, bk, bv = _extremes(fmt)
    L, T, C_ = k.shape
    if fmt == 3:
        ref = oracle_mod.compress_v3(k, v, Tc, bk, bv, group=G)
        side_ref = ref["side"]
    else:
        ref = oracle_mod.compress_ex(k, v, Tc, bk, bv, fmt=fmt, group=G)
        side_ref = ref["cdf" if fmt == 1 else "rec"]
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=fmt, group=G)
    out = cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    ok, ov = cd.decompress()
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0 and int(cd.dstatus.item()) == 0
    assert np.array_equal(out.max1.cpu().numpy().view(np.uint16), ref["max1"])
    if fmt == 1:
        side = out.cdf[:side_ref.size].cpu().numpy().view(np.uint16)
    elif fmt == 2:
        side = out.rec[:side_ref.size].cpu().numpy()
    else:
        assert out.side3_bytes() == side_ref.size
        side = out.side3[:side_ref.size].cpu().numpy()
    assert np.array_equal(side, side_ref)
    ns = 2 * L * T
    assert np.array_equal(out.len[:ns].cpu().numpy().view(np.uint32), ref["len"])
    assert np.array_equal(out.off.cpu().numpy().view(np.uint64), ref["off"])
    total = int(ref["off"][-1])
    assert np.array_equal(out.packed[:total].cpu().numpy(), ref["packed"])
    if fmt == 3:
        wk, wv = oracle_mod.decompress_v3(ref["packed"], ref["len"], ref["side"], ref["max1"], L, T, C_, Tc,
                                          bk, bv, group=G)
    else:
        wk, wv = oracle_mod.decompress_ex(ref["packed"], ref["off"], ref["len"], side_ref, ref["max1"], L, T, C_,
                                          Tc, bk, bv, fmt=fmt, group=G)
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), wk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), wv.view(np.uint32))
    # the degenerate layers decode to what the method says, whatever the format
    if G == 1:
        assert not ok[0].any()                                   # max1 = 0 -> 0
        assert bool((ov[0] == 1.0).all())                        # constant 1 -> +max1
        assert torch.equal(ov[2].cpu(), torch.from_numpy(v[2].astype(np.float32)))  # -c rows -> -max1
