"""Full-size workloads (the 34B-shaped 32K-token context and the 80K-token
low-locality stress case) on the GPU, in the launch configuration the
benchmark times (one compress and one decompress call over the whole tensor),
in all three side-information formats.

The oracle cannot code 6-10 GB in a test at once, so:
- whole chunks (the first, the last and 14 drawn at random) are coded by the
  oracle, one spawned process per chunk, from inputs the host generator
  produces on its own (the whole tensor for AR(1) workloads, whose chunks
  cost their token prefix to generate alone; each chunk alone otherwise), and every output of those chunks (max1, the side
  information block, stream lengths, packed bytes, dequantised values) must
  match the GPU's bit for bit, in all three side-information formats;
- sampled (chunk, kv, layer) slices are also coded alone by the oracle and
  compared the same way (formats 1 and 2);
- properties that hold at any size are checked over every element on the GPU:
  status words clear, offsets the exclusive scan of the lengths, lengths within
  2C + 8, and the quantisation error bound |x - x^| <= max1/(2 MAX) + ulp(max1).
"""
import hashlib
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle_chunks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from kv_cache_compression_cg_gb300 import build, codec
    build.build()
    return codec


def _samples(w, seed):
    nch = w.n_chunks
    rng = np.random.default_rng(seed)
    picks = [(0, 0, 0), (nch - 1, 1, w.L - 1), (nch // 2, 0, w.L // 2), (nch // 3, 1, 1)]
    for _ in range(2):
        picks.append((int(rng.integers(nch)), int(rng.integers(2)), int(rng.integers(w.L))))
    return picks


def _check_slice(cg, oracle_mod, synth_mod, w, k, v, codec, out, ok, ov, kc, kv, l, fmt, host=None):
    L, T, C_, Tc = w.L, w.T, w.C, w.chunk_tokens
    bins = (w.bins_k, w.bins_v)[kv]
    A_k, A_v = max(w.bins_k), max(w.bins_v)
    A = (A_k, A_v)[kv]
    t0, t1 = kc * Tc, min(T, (kc + 1) * Tc)
    Tk = t1 - t0
    x = host[kv][l, t0:t1] if host is not None else synth_mod.generate_slice_range(w, kv, l, t0, t1)
    dev_x = (k, v)[kv][l, t0:t1].cpu().numpy()
    assert np.array_equal(dev_x.view(np.uint16), x.view(np.uint16)), "device generator differs from host"
    # the oracle on [2 layers][Tk][C]: layer 0 is the slice, layer 1 a zero
    # layer with bins A, so that format 1's alphabet is the tensor's A (format
    # 2's alphabets are per layer)
    K = np.zeros((2, Tk, C_), np.float16)
    K[0] = x
    V = np.zeros((2, Tk, C_), np.float16)
    if fmt == 1:
        ref = oracle_mod.compress(K, V, Tc, [bins[l], A], [A, A])
        assert ref["A_k"] == A
    else:
        ref = oracle_mod.compress_v2(K, V, Tc, [bins[l], A], [A, A])
    # max1
    got_m1 = out.max1[kv, l, t0:t1].cpu().numpy().view(np.uint16)
    assert np.array_equal(got_m1, ref["max1"][0, 0])
    # side information of the slice: CDF rows or count records
    if fmt == 1:
        g0 = oracle_mod.cdf_offset(L, C_, A_k, A_v, kc, kv, l, 0)
        got_cdf = out.cdf[g0:g0 + C_ * A].cpu().numpy().view(np.uint16)
        assert np.array_equal(got_cdf, ref["cdf"][:C_ * A])
    else:
        Al = oracle_mod.alphabet_v2(bins[l])
        g0 = oracle_mod.rec_offset(L, C_, w.bins_k, w.bins_v, kc, kv, l, 0)
        got_rec = out.rec[g0:g0 + C_ * Al].cpu().numpy()
        assert np.array_equal(got_rec, ref["rec"][:C_ * Al])
    # stream lengths and bytes
    s0 = oracle_mod.stream_id(L, T, Tc, kc, kv, l, 0)
    got_len = out.len[s0:s0 + Tk].cpu().numpy().view(np.uint32)
    assert np.array_equal(got_len, ref["len"][:Tk])
    b0, b1 = int(out.off[s0].item()), int(out.off[s0 + Tk].item())
    assert b1 - b0 == int(ref["off"][Tk])
    assert np.array_equal(out.packed[b0:b1].cpu().numpy(), ref["packed"][:b1 - b0])
    # dequantised output of the slice
    if fmt == 1:
        rk, _ = oracle_mod.decompress(ref["packed"], ref["off"], ref["len"], ref["cdf"], ref["max1"],
                                      2, Tk, C_, Tc, [bins[l], A], [A, A])
    else:
        rk, _ = oracle_mod.decompress_v2(ref["packed"], ref["off"], ref["len"], ref["rec"], ref["max1"],
                                         2, Tk, C_, Tc, [bins[l], A], [A, A])
    got = (ok, ov)[kv][l, t0:t1].cpu().numpy()
    assert np.array_equal(got.view(np.uint32), rk[0].view(np.uint32))


def _check_properties(w, k, v, codec, out, ok, ov):
    ns = 2 * w.L * w.T
    ln = out.len[:ns].to(torch.int64) & 0xFFFFFFFF
    off = out.off
    assert int(off[0].item()) == 0
    assert torch.equal(off[1:] - off[:-1], ln)
    assert int(ln.max().item()) <= 2 * w.C + 8
    assert int(off[-1].item()) <= codec.capacity
    for kv, (x, xh, bins) in enumerate(((k, ok, w.bins_k), (v, ov, w.bins_v))):
        for l in range(w.L):
            m1 = out.max1[kv, l].view(torch.float16)
            ulp = (out.max1[kv, l] + 1).view(torch.float16).float() - m1.float()
            MAX = bins[l] // 2 - 1
            bound = m1.float() / (2 * MAX) + ulp
            err = (xh[l] - x[l].float()).abs().amax(dim=1)
            assert bool((err <= bound).all()), f"error bound broken at kv={kv} layer={l}"


def _chunk_picks(w, seed, n=14):
    """The first and last chunks and n distinct others drawn at random."""
    nch = w.n_chunks
    inner = np.arange(1, nch - 1)
    rng = np.random.default_rng(seed)
    mid = rng.choice(inner, size=min(n, inner.size), replace=False) if inner.size else []
    return sorted({0, nch - 1, *(int(c) for c in mid)})


def _check_chunk(oracle_mod, w, out, ok, ov, rec_all, ref, fmt):
    L, T, C_, Tc = w.L, w.T, w.C, w.chunk_tokens
    kc = ref["kc"]
    t0, t1 = kc * Tc, min(T, (kc + 1) * Tc)
    Tk = t1 - t0
    assert np.array_equal(out.max1[:, :, t0:t1].cpu().numpy().view(np.uint16), ref["max1"]), kc
    side = ref["side"]
    if fmt == 1:
        g0 = oracle_mod.cdf_offset(L, C_, max(w.bins_k), max(w.bins_v), kc, 0, 0, 0)
        got = out.cdf[g0:g0 + side.size].cpu().numpy().view(np.uint16)
    else:
        g0 = oracle_mod.rec_offset(L, C_, w.bins_k, w.bins_v, kc, 0, 0, 0)
        got = out.rec[g0:g0 + side.size].cpu().numpy() if fmt == 2 else rec_all[g0:g0 + side.size]
    assert np.array_equal(got, side), kc
    s0 = oracle_mod.stream_id(L, T, Tc, kc, 0, 0, 0)
    ns = 2 * L * Tk
    assert np.array_equal(out.len[s0:s0 + ns].cpu().numpy().view(np.uint32), ref["len"]), kc
    b0, b1 = int(out.off[s0].item()), int(out.off[s0 + ns].item())
    assert b1 - b0 == ref["packed"].size, kc
    assert np.array_equal(out.packed[b0:b1].cpu().numpy(), ref["packed"]), kc
    h = hashlib.sha256()
    h.update(ok[:, t0:t1].contiguous().cpu().numpy().tobytes())
    h.update(ov[:, t0:t1].contiguous().cpu().numpy().tobytes())
    assert h.hexdigest() == ref["out_sha256"], kc


_HOST = {}


def _host_tensor(synth_mod, w):
    """The host generator's whole K, V for w, kept for the next format's test
    of the same workload (one workload at a time)."""
    if w.name not in _HOST:
        _HOST.clear()
        _HOST[w.name] = synth_mod.generate(w)
    return _HOST[w.name]


@pytest.mark.parametrize("fmt", [1, 2, 3])
@pytest.mark.parametrize("name", ["ctx32k", "stress80k"])
def test_fullsize_sampled_parity_and_properties(cg, oracle_mod, synth_mod, name, fmt):
    w = synth_mod.WORKLOADS[name]
    picks = _chunk_picks(w, seed=len(name) + fmt)
    # An AR(1) chunk generated alone costs its whole token prefix: generate the
    # tensor once on the host (all cores) and hand each worker its chunk. An
    # iid workload's chunks are cheap alone.
    host = _host_tensor(synth_mod, w) if w.kind == synth_mod.AR1 else _HOST.clear()

    def job(kc):
        if host is None:
            return (name, kc, fmt)
        t0, t1 = kc * w.chunk_tokens, min(w.T, (kc + 1) * w.chunk_tokens)
        return (name, kc, fmt, None, host[0][:, t0:t1].copy(), host[1][:, t0:t1].copy())

    # the oracle's chunks run on the host cores while the GPU codes the tensor
    pool = mp.get_context("spawn").Pool(processes=min(len(picks), os.cpu_count() or 1))
    try:
        pending = pool.starmap_async(oracle_chunks.code_chunk, [job(kc) for kc in picks])
        k, v = synth_mod.generate_device(w)
        codec = cg.Codec(w.L, w.T, w.C, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens,
                         capacity=w.elements // 2, fmt=fmt)
        out = codec.compress(k, v)
        ok, ov = codec.decompress()
        torch.cuda.synchronize()
        assert int(out.status.item()) == 0
        assert int(codec.dstatus.item()) == 0
        _check_properties(w, k, v, codec, out, ok, ov)
        rec_all = None
        if fmt == 3:  # the whole side buffer must parse; its records are compared per chunk
            side = out.side3[:out.side3_bytes()].cpu().numpy()
            rec_all = oracle_mod.v3_to_records(side, w.L, w.T, w.C, w.chunk_tokens, w.bins_k, w.bins_v)
        else:
            for kc, kv, l in _samples(w, seed=len(name)):
                _check_slice(cg, oracle_mod, synth_mod, w, k, v, codec, out, ok, ov, kc, kv, l, fmt, host)
        refs = pending.get(timeout=1800)
    finally:
        pool.close()
        pool.join()
    assert [r["kc"] for r in refs] == picks
    for ref in refs:
        _check_chunk(oracle_mod, w, out, ok, ov, rec_all, ref, fmt)
