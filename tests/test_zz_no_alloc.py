"""cg_compress_chunk_noalloc: the compress entry point for callers that cannot
allocate device memory (a host framework's pool owns all device memory, or the
path must not synchronise on cudaMalloc). It must produce exactly what
cg_compress_chunk produces with a caller-provided workspace, call after call,
although every call reuses the same static scratch inside the library.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test first. It also passes on its own, in a fresh
process."""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _ptr(t):
    return C.c_void_p(t.data_ptr())


def _bins(b):
    a = np.ascontiguousarray(np.asarray(b, np.int32))
    return a, C.c_void_p(a.ctypes.data)


def _outputs(lib, shp, pk, pv, capacity):
    ns = int(lib.cg_num_streams(C.byref(shp)))
    ncdf = int(lib.cg_cdf_elems(C.byref(shp), pk, pv))
    return {
        "max1": torch.full((2, shp.L, shp.T), -1, dtype=torch.int16, device="cuda"),
        "cdf": torch.full((ncdf,), -1, dtype=torch.int16, device="cuda"),
        "packed": torch.full((capacity,), 0xEE, dtype=torch.uint8, device="cuda"),
        "len": torch.full((ns,), -1, dtype=torch.int32, device="cuda"),
        "off": torch.full((ns + 1,), -1, dtype=torch.int64, device="cuda"),
        "status": torch.zeros(1, dtype=torch.int32, device="cuda"),
    }


def _compare(a, b):
    total = int(a["off"][-1].item())
    assert total == int(b["off"][-1].item())
    for key in ("max1", "cdf", "len", "off", "status"):
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(a["packed"][:total], b["packed"][:total])
    assert int(a["status"].item()) == 0


def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    from kv_cache_compression_cg_gb300 import build, capi, synth
    build.build()
    lib = capi.load()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)

    # three different shapes in a row: each call runs on whatever the one before
    # left in the shared static scratch. The last has 13 channels, so the library
    # takes its multi-kernel path (quantise, count-and-code, scan and pack), which
    # carves the symbol tensor and the scan partials out of the same scratch.
    rng = np.random.default_rng(3)
    odd = (rng.standard_normal((3, 300, 13)) * rng.lognormal(0, 0.5, (1, 1, 13))).astype(np.float16)
    cases = [(*synth.generate(synth.WORKLOADS[n]), synth.WORKLOADS[n]) for n in ("mistral_chunk", "tiny")]
    cases.append((odd, -odd[:, ::-1].copy(), None))
    for k_h, v_h, w in cases:
        k = torch.from_numpy(k_h).cuda()
        v = torch.from_numpy(v_h).cuda()
        L, T, C_ = k_h.shape
        Tc = w.chunk_tokens if w is not None else 128
        shp = capi.cg_shape(L, T, C_, Tc, T * C_)
        bk, pk = _bins(w.bins_k if w is not None else [32, 16, 8])
        bv, pv = _bins(w.bins_v if w is not None else [16, 16, 32])
        cap = int(lib.cg_max_compressed_bytes(C.byref(shp)))
        need = int(lib.cg_compress_workspace_bytes(C.byref(shp)))
        assert 0 < need <= capi.CG_NOALLOC_WORKSPACE_BYTES

        ref = _outputs(lib, shp, pk, pv, cap)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        rc = lib.cg_compress_chunk(_ptr(k), _ptr(v), C.byref(shp), pk, pv, _ptr(ref["max1"]),
                                   _ptr(ref["cdf"]), _ptr(ref["packed"]), cap, _ptr(ref["len"]),
                                   _ptr(ref["off"]), _ptr(ws), need, _ptr(ref["status"]), stream)
        assert rc == 0

        got = _outputs(lib, shp, pk, pv, cap)
        rc = lib.cg_compress_chunk_noalloc(_ptr(k), _ptr(v), C.byref(shp), pk, pv,
                                           _ptr(got["max1"]), _ptr(got["cdf"]),
                                           _ptr(got["packed"]), cap, _ptr(got["len"]),
                                           _ptr(got["off"]), _ptr(got["status"]), stream)
        assert rc == 0
        torch.cuda.synchronize()
        _compare(got, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    from kv_cache_compression_cg_gb300 import build, capi
    build.build()
    lib = capi.load()
    shp = capi.cg_shape(32, 4096, 1024, 256, 4096 * 1024)  # needs far more than 64 MiB
    assert int(lib.cg_compress_workspace_bytes(C.byref(shp))) > capi.CG_NOALLOC_WORKSPACE_BYTES
    bk, pk = _bins([16] * 32)
    fake = C.c_void_p(0x100000)  # never touched: the size check comes first
    rc = lib.cg_compress_chunk_noalloc(fake, fake, C.byref(shp), pk, None, fake, fake, fake, 1, fake,
                                       fake, None, None)
    assert rc == capi.CG_ERR_WORKSPACE
