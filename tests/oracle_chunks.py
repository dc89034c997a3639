"""The oracle over whole chunks of a workload, one chunk per call, for a pool
of spawned processes: each call regenerates its chunk with the host generator
and returns what the GPU's outputs for that chunk must equal.

Chunks are independent (their own symbol statistics, their own streams), so a
chunk coded alone as a one-chunk tensor gives exactly that chunk's block of
the whole tensor's outputs: max1 [2][L][Tk], the side information block, the
stream lengths, the streams' bytes, and the dequantised values (returned as a
SHA-256 of K's then V's binary32 bytes, to keep what crosses the process
boundary small)."""
from __future__ import annotations

import hashlib

import numpy as np


def code_chunk(name: str, kc: int, fmt: int, T: int | None = None, k=None, v=None) -> dict:
    """Chunk kc of workload `name` (its first T tokens if T is given) in
    side-information format fmt. k, v: the chunk's host-generated values
    [L][Tk][C] when the caller has them (an AR(1) workload's late chunks cost
    their whole token prefix to generate alone)."""
    import oracle
    from kv_cache_compression_cg_gb300 import synth
    w = synth.WORKLOADS[name]
    Tc = w.chunk_tokens
    T = w.T if T is None else T
    t0, t1 = kc * Tc, min(T, (kc + 1) * Tc)
    Tk = t1 - t0
    if k is None:
        k = np.stack([synth.generate_slice_range(w, 0, l, t0, t1) for l in range(w.L)])
        v = np.stack([synth.generate_slice_range(w, 1, l, t0, t1) for l in range(w.L)])
    assert k.shape == v.shape == (w.L, Tk, w.C)
    bk, bv = w.bins_k, w.bins_v
    if fmt == 1:
        r = oracle.compress(k, v, Tc, bk, bv)
        side = r["cdf"]
        dk, dv = oracle.decompress(r["packed"], r["off"], r["len"], r["cdf"], r["max1"], w.L, Tk, w.C, Tc, bk, bv)
    elif fmt == 2:
        r = oracle.compress_v2(k, v, Tc, bk, bv)
        side = r["rec"]
        dk, dv = oracle.decompress_v2(r["packed"], r["off"], r["len"], r["rec"], r["max1"], w.L, Tk, w.C, Tc,
                                      bk, bv)
    else:
        r = oracle.compress_v3(k, v, Tc, bk, bv)
        side = oracle.v3_to_records(r["side"], w.L, Tk, w.C, Tc, bk, bv)
        dk, dv = oracle.decompress_v3(r["packed"], r["len"], r["side"], r["max1"], w.L, Tk, w.C, Tc, bk, bv)
    h = hashlib.sha256()
    h.update(np.ascontiguousarray(dk).tobytes())
    h.update(np.ascontiguousarray(dv).tobytes())
    total = int(r["off"][-1])
    return {"kc": kc, "max1": r["max1"], "side": side, "len": r["len"], "packed": r["packed"][:total],
            "out_sha256": h.hexdigest()}
