"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every function include/cachegen.h declares, its size helpers
agree with the oracle's layout, and bad arguments are rejected on the host
before any device work."""
import ctypes as C

import numpy as np
import pytest


@pytest.fixture(scope="module")
def lib():
    from kv_cache_compression_cg_gb300 import build, capi
    build.build()
    return capi.load()


def test_exports_every_declared_function(lib):
    from kv_cache_compression_cg_gb300 import capi
    names = capi.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), f"{n} declared in cachegen.h but not exported"
        assert n in capi.SIGNATURES, f"{n} has no binding"


def test_version(lib):
    assert lib.cg_version().decode().startswith("cachegen-gb300 formats-1,2")


def _shape(L, T, C_, Tc=256, ls=None):
    from kv_cache_compression_cg_gb300 import capi
    return capi.cg_shape(L, T, C_, Tc, T * C_ if ls is None else ls)


def _b(x):
    a = np.ascontiguousarray(np.asarray(x, np.int32))
    return a, C.c_void_p(a.ctypes.data)


@pytest.mark.parametrize("L,T,C_,Tc,bk,bv", [
    (2, 64, 64, 64, [32, 16], [32, 16]),
    (3, 150, 40, 64, [32, 16, 8], [4, 16, 255]),
    (32, 4096, 1024, 256, [32] * 10 + [16] * 22, None),
    (48, 32768, 1024, 256, [32] * 16 + [16] * 32, None),
])
def test_sizes_match_oracle_layout(lib, oracle_mod, L, T, C_, Tc, bk, bv):
    s = _shape(L, T, C_, Tc)
    ak, pk = _b(bk)
    av, pv = _b(bv if bv is not None else bk)
    assert lib.cg_num_streams(C.byref(s)) == oracle_mod.num_streams(L, T)
    A_k, A_v = oracle_mod.alphabet(ak), oracle_mod.alphabet(av)
    assert lib.cg_cdf_elems(C.byref(s), pk, pv) == oracle_mod.cdf_elems(L, T, C_, Tc, A_k, A_v)
    if bv is None:
        assert lib.cg_cdf_elems(C.byref(s), pk, None) == oracle_mod.cdf_elems(L, T, C_, Tc, A_k, A_k)
    assert lib.cg_max_compressed_bytes(C.byref(s)) == oracle_mod.max_compressed_bytes(L, T, C_)
    ws = lib.cg_workspace_bytes(C.byref(s))
    assert ws >= 2 * L * T * (2 * C_ + 8) and ws % 256 == 0
    assert lib.cg_compress_workspace_bytes(C.byref(s)) >= ws + 2 * L * T * C_


@pytest.mark.parametrize("bad", [
    dict(L=0), dict(L=1025), dict(T=-1), dict(C=0), dict(C=65537), dict(Tc=0), dict(Tc=1025),
    dict(ls=10),
])
def test_invalid_shapes_rejected(lib, bad):
    L, T, C_, Tc, ls = bad.get("L", 2), bad.get("T", 64), bad.get("C", 64), bad.get("Tc", 64), None
    if "ls" in bad:
        ls = bad["ls"]
    s = _shape(L, T, C_, Tc, ls)
    assert lib.cg_num_streams(C.byref(s)) == 0
    assert lib.cg_workspace_bytes(C.byref(s)) == 0
    b, pb = _b([16] * max(L, 1))
    fake = C.c_void_p(0x1000)  # never dereferenced: validation fails first
    assert lib.cg_quantize(fake, fake, C.byref(s), pb, None, fake, fake, None, None) == 1


@pytest.mark.parametrize("bins", [[3, 16], [16, 257], [0, 16], [-8, 16]])
def test_invalid_bins_rejected(lib, bins):
    s = _shape(2, 64, 64, 64)
    b, pb = _b(bins)
    fake = C.c_void_p(0x1000)
    assert lib.cg_cdf_elems(C.byref(s), pb, None) == 0
    assert lib.cg_quantize(fake, fake, C.byref(s), pb, None, fake, fake, None, None) == 1
    ok, pok = _b([16, 16])
    assert lib.cg_quantize(fake, fake, C.byref(s), pok, pb, fake, fake, None, None) == 1


def test_null_and_misaligned_pointers_rejected(lib):
    s = _shape(2, 64, 64, 64)
    b, pb = _b([16, 16])
    fake = C.c_void_p(0x1000)
    odd = C.c_void_p(0x1001)
    assert lib.cg_quantize(None, fake, C.byref(s), pb, None, fake, fake, None, None) == 1
    assert lib.cg_quantize(odd, fake, C.byref(s), pb, None, fake, fake, None, None) == 1
    ws_odd = C.c_void_p(0x1010)
    assert lib.cg_encode(fake, fake, C.byref(s), pb, None, fake, 100, fake, fake, ws_odd, 1 << 40,
                         None, None) == 1  # workspace not 256-byte aligned
    ws = C.c_void_p(0x10000)
    assert lib.cg_encode(fake, fake, C.byref(s), pb, None, fake, 100, fake, fake, ws, 16,
                         None, None) == 2  # workspace too small
    assert lib.cg_decode(odd, 10, fake, fake, fake, C.byref(s), pb, None, fake, None, None) == 1
    assert lib.cg_decompress_chunk(fake, 10, fake, fake, fake, fake, C.byref(s), pb, None, odd, fake,
                                   None, None) == 1
    assert lib.cg_compress_chunk(fake, fake, C.byref(s), pb, None, fake, fake, fake, 10, fake, None,
                                 ws, 1 << 40, None, None) == 1  # off is required


def test_serving_layout_arguments_rejected(lib):
    """cg_decompress_chunk_ex rejects, before touching the device: unknown
    format or output type, a layer stride below T*C, chunks over 256 tokens,
    outputs not aligned to their element size."""
    s = _shape(2, 64, 64, 64)
    b, pb = _b([16, 16])
    fake = C.c_void_p(0x1000)
    odd = C.c_void_p(0x1001)
    ls = 64 * 64

    def call(shape, fmt, dtype, ok, ov, stride, group=1):
        return lib.cg_decompress_chunk_ex(fake, 10, fake, fake, fake, fake, C.byref(shape), pb, None, fmt, group,
                                          dtype, ok, ov, stride, None, None)
    assert call(s, 3, 0, fake, fake, ls) == 1
    assert call(s, 1, 2, fake, fake, ls) == 1
    assert call(s, 2, 1, fake, fake, ls - 1) == 1
    assert call(_shape(2, 600, 64, 300), 1, 0, fake, fake, 600 * 64) == 1
    assert call(s, 1, 1, odd, fake, ls) == 1
    assert call(s, 2, 0, fake, C.c_void_p(0x1002), ls) == 1
    assert call(s, 1, 0, None, fake, ls) == 1
    assert call(s, 1, 0, fake, fake, ls, group=0) == 1
    assert call(s, 1, 0, fake, fake, ls, group=1025) == 1


def test_delta_arguments_rejected(lib):
    """The token-locality delta's entry points reject a group outside
    [1, 1024], an unknown format and format 2 with chunks over 256 tokens,
    before touching the device."""
    s = _shape(2, 64, 64, 64)
    b, pb = _b([16, 16])
    fake = C.c_void_p(0x1000)
    ws = C.c_void_p(0x10000)
    for g in (0, -3, 1025):
        assert lib.cg_quantize_delta(fake, fake, C.byref(s), pb, None, g, fake, fake, None, None) == 1
        assert lib.cg_dequantize_delta(fake, fake, C.byref(s), pb, None, g, fake, fake, None, None) == 1
        assert lib.cg_compress_chunk_ex(fake, fake, C.byref(s), pb, None, 1, g, fake, fake, fake, 10, fake, fake,
                                        ws, 1 << 40, None, None) == 1
    assert lib.cg_compress_chunk_ex(fake, fake, C.byref(s), pb, None, 3, 4, fake, fake, fake, 10, fake, fake,
                                    ws, 1 << 40, None, None) == 1
    big = _shape(2, 600, 64, 300)
    assert lib.cg_compress_chunk_ex(fake, fake, C.byref(big), pb, None, 2, 4, fake, fake, fake, 10, fake, fake,
                                    ws, 1 << 40, None, None) == 1
    assert lib.cg_compress_chunk_ex(fake, fake, C.byref(s), pb, None, 1, 4, fake, fake, fake, 10, fake, fake,
                                    ws, 16, None, None) == 2  # workspace too small


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from kv_cache_compression_cg_gb300 import capi
    monkeypatch.setattr(capi, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(capi, "_LIB", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        capi.load()


def test_record_bytes_match_oracle(oracle_mod):
    from kv_cache_compression_cg_gb300 import capi, codec
    import numpy as np
    lib = capi.load()
    for L, T, C_, Tc, bk, bv in [(2, 64, 64, 64, [32, 16], [16, 32]), (3, 200, 40, 64, [32, 16, 7], [8, 8, 256]),
                                (1, 300, 8, 256, [4], [5])]:
        shp = codec.make_shape(L, T, C_, Tc)
        bka, bva = np.array(bk, np.int32), np.array(bv, np.int32)
        got = lib.cg_record_bytes(ctypes_ref(shp), bka.ctypes.data, bva.ctypes.data)
        assert got == oracle_mod.rec_bytes(L, T, C_, Tc, bk, bv)
    shp = codec.make_shape(1, 600, 8, 300)  # format 2 needs chunks of at most 256 tokens
    b = np.array([16], np.int32)
    assert lib.cg_record_bytes(ctypes_ref(shp), b.ctypes.data, b.ctypes.data) == 0


def ctypes_ref(x):
    import ctypes
    return ctypes.byref(x)


def test_format3_sizes_and_rejections(oracle_mod):
    """Format 3's sizes equal the oracle's; arguments the library cannot
    serve are refused before touching the device."""
    from kv_cache_compression_cg_gb300 import capi, codec
    import ctypes
    import numpy as np
    lib = capi.load()
    for L, T, C_, Tc, bk, bv in [(2, 64, 64, 64, [32, 16], [16, 32]), (3, 200, 40, 64, [32, 16, 7], [8, 8, 33]),
                                (1, 300, 8, 256, [4], [5])]:
        shp = codec.make_shape(L, T, C_, Tc)
        bka, bva = np.array(bk, np.int32), np.array(bv, np.int32)
        assert lib.cg_side3_fixed_bytes(ctypes.byref(shp)) == oracle_mod.v3_fixed_bytes(L, T, C_, Tc)
        assert lib.cg_side3_max_bytes(ctypes.byref(shp), bka.ctypes.data, bva.ctypes.data) == \
            oracle_mod.v3_max_bytes(L, T, C_, Tc, bk, bv)
    wide = np.array([64], np.int32)  # A = 63: past a 32-bit presence mask
    shp = codec.make_shape(1, 64, 8, 64)
    assert lib.cg_side3_max_bytes(ctypes.byref(shp), wide.ctypes.data, wide.ctypes.data) == 0
    long_chunks = codec.make_shape(1, 600, 8, 300)
    b = np.array([16], np.int32)
    assert lib.cg_side3_max_bytes(ctypes.byref(long_chunks), b.ctypes.data, b.ctypes.data) == 0
    fake, ws = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x10000)
    need = lib.cg_side3_max_bytes(ctypes.byref(shp), b.ctypes.data, b.ctypes.data)
    assert lib.cg_compress_chunk_v3(fake, fake, ctypes.byref(shp), b.ctypes.data, None, 1, fake, fake, need - 1, fake,
                                    100, fake, fake, ws, 1 << 40, None, None) == 1  # side buffer too small
    assert lib.cg_compress_chunk_v3(fake, fake, ctypes.byref(shp), b.ctypes.data, None, 1, fake, fake, need, fake,
                                    100, fake, fake, ws, 16, None, None) == 2  # workspace too small
    fixed = lib.cg_side3_fixed_bytes(ctypes.byref(shp))
    assert lib.cg_decompress_chunk_v3(fake, 100, fake, fake, fixed - 1, fake, ctypes.byref(shp), b.ctypes.data, None,
                                      1, 0, fake, fake, 64 * 8, ws, 1 << 40, None, None) == 1  # shorter than its fixed part
