"""Out-of-bounds write check for every entry point (compute-sanitizer stands in
for nothing here: each output buffer is followed by canary bytes).

Every output a call writes is carved from a larger device allocation whose
bytes all hold a position-dependent pattern before the call. After the call:
  - the bytes past the output's extent (256 of them) still hold the pattern;
  - outputs whose written extent is data-dependent (packed bytes up to
    off[nstreams], the format 3 side buffer up to its size) keep the pattern
    from that extent to the end of the allocation;
  - strided outputs ([L, 2, T, C] caches with a gap after every plane) keep
    the pattern in the gaps.
The same calls on plain allocations give identical outputs, so the guarded
runs did the real work."""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

PAD = 256


@pytest.fixture(scope="module")
def cg():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from kv_cache_compression_cg_gb300 import build, codec
    build.build()
    return codec


def _pattern(n: int) -> torch.Tensor:
    return torch.from_numpy(((np.arange(n, dtype=np.int64) * 37 + 11) % 251).astype(np.uint8)).cuda()


class Guarded:
    """One allocation: `n` bytes of output then PAD canary bytes, all patterned."""

    def __init__(self, n: int, dtype=torch.uint8, shape=None):
        self.n = int(n)
        self.raw = _pattern(self.n + PAD)
        esz = torch.tensor([], dtype=dtype).element_size()
        assert self.n % esz == 0
        body = self.raw[:self.n].view(dtype)
        self.t = body.view(shape) if shape is not None else body

    def check(self, written: int | None = None, what: str = "") -> None:
        """Bytes from `written` (default: the output's extent) to the end
        still hold the pattern."""
        start = self.n if written is None else int(written)
        ref = _pattern(self.n + PAD)
        got = self.raw[start:]
        bad = (got != ref[start:]).nonzero()
        assert bad.numel() == 0, f"{what}: byte {start + int(bad[0])} past the extent was written"


def _case(synth_mod, name):
    if name in ("tiny", "mistral_chunk"):
        w = synth_mod.WORKLOADS[name]
        k, v = synth_mod.generate(w)
        return k, v, w.chunk_tokens, list(w.bins_k), list(w.bins_v)
    rng = np.random.default_rng(len(name) + 7)
    shapes = {"ragged": (3, 150, 40, 64, [32, 16, 8], [4, 16, 255]),   # wide alphabet: the step path
              "odd_c": (2, 70, 13, 64, [16, 32], [8, 33]),             # C % 8 != 0: the step path
              "long_chunk": (2, 1300, 24, 600, [255, 16], [32, 8]),    # chunks of 600 tokens, format 1
              "bins64": (3, 300, 136, 256, [64, 40, 16], [33, 64, 8]),  # the 64-symbol fused kernel
              "bins20": (2, 300, 40, 128, [20, 12], [12, 20]),         # format-1 rows of 20 entries
              "bins24_36": (2, 260, 64, 256, [24, 16], [36, 10])}      # rows of 24 (16-byte stores) and 36
    L, T, C_, Tc, bk, bv = shapes[name]
    k = (rng.standard_normal((L, T, C_)) * rng.lognormal(0, 0.5, (1, 1, C_))).astype(np.float16)
    v = rng.standard_t(3, size=(L, T, C_)).astype(np.float16)
    return k, v, Tc, bk, bv


def _guard_codec(cd):
    """Swap every buffer a Codec passes to the library for a guarded one."""
    o = cd.out
    g = {}

    def swap(name, t):
        gg = Guarded(t.numel() * t.element_size(), t.dtype, tuple(t.shape))
        g[name] = gg
        return gg.t

    o.max1 = swap("max1", o.max1)
    o.cdf = swap("cdf", o.cdf)
    o.packed = swap("packed", o.packed)
    o.len = swap("len", o.len)
    o.off = swap("off", o.off)
    o.status = swap("status", o.status)
    o.status.zero_()
    if o.rec is not None:
        o.rec = swap("rec", o.rec)
    if o.side3 is not None:
        o.side3 = swap("side3", o.side3)
    cd.workspace = swap("workspace", cd.workspace)
    cd.out_k = swap("out_k", cd.out_k)
    cd.out_v = swap("out_v", cd.out_v)
    cd.dstatus = swap("dstatus", cd.dstatus)
    cd.dstatus.zero_()
    return g


CASES = [("tiny", 1, 1), ("tiny", 2, 1), ("tiny", 3, 1), ("mistral_chunk", 2, 1), ("mistral_chunk", 2, 10),
         ("mistral_chunk", 3, 10), ("mistral_chunk", 1, 4), ("ragged", 1, 1), ("ragged", 2, 1), ("odd_c", 2, 1),
         ("odd_c", 3, 10), ("long_chunk", 1, 1), ("bins64", 1, 1), ("bins64", 2, 10), ("bins20", 1, 1),
         ("bins24_36", 1, 1)]


@pytest.mark.parametrize("name,fmt,group", CASES)
def test_compress_decompress_write_nothing_past_their_outputs(cg, synth_mod, name, fmt, group):
    k, v, Tc, bk, bv = _case(synth_mod, name)
    L, T, C_ = k.shape
    kt, vt = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    plain = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=fmt, group=group)
    po = plain.compress(kt, vt)
    pk, pv = plain.decompress()
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=fmt, group=group)
    g = _guard_codec(cd)
    out = cd.compress(kt, vt)
    ok, ov = cd.decompress()
    torch.cuda.synchronize()
    assert int(out.status.item()) == 0 and int(cd.dstatus.item()) == 0
    total = out.total_bytes()
    assert total == po.total_bytes()
    assert torch.equal(out.packed[:total], po.packed[:total])
    assert torch.equal(out.len, po.len) and torch.equal(out.off, po.off) and torch.equal(out.max1, po.max1)
    assert torch.equal(ok.view(torch.int32), pk.view(torch.int32))
    assert torch.equal(ov.view(torch.int32), pv.view(torch.int32))
    g["packed"].check(total, "packed past off[nstreams]")
    if fmt == 3:
        n3 = out.side3_bytes()
        assert torch.equal(out.side3[:n3], po.side3[:n3])
        g["side3"].check(n3, "format 3 side buffer past its size")
    elif fmt == 2:
        assert torch.equal(out.rec, po.rec)
    else:
        assert torch.equal(out.cdf, po.cdf)
    for name_, gg in g.items():
        if name_ not in ("packed", "side3"):
            gg.check(what=name_)


@pytest.mark.parametrize("name,fmt,dtype", [("tiny", 1, torch.float16), ("mistral_chunk", 2, torch.float16),
                                            ("mistral_chunk", 3, torch.float32), ("odd_c", 2, torch.float16)])
def test_serving_layout_gaps_stay_untouched(cg, synth_mod, name, fmt, dtype):
    """[L, 2, T + 1, C] cache: K and V planes of T rows with one spare row
    after each; the spare rows and the bytes after the cache keep the pattern."""
    k, v, Tc, bk, bv = _case(synth_mod, name)
    L, T, C_ = k.shape
    cd = cg.Codec(L, T, C_, bk, bv, chunk_tokens=Tc, fmt=fmt)
    cd.compress(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())
    esz = torch.tensor([], dtype=dtype).element_size()
    g = Guarded(L * 2 * (T + 1) * C_ * esz, dtype, (L, 2, T + 1, C_))
    cd.decompress_into(g.t[:, 0, :T], g.t[:, 1, :T])
    torch.cuda.synchronize()
    assert int(cd.dstatus.item()) == 0
    ref = _pattern(g.n + PAD)
    spare = g.raw[:g.n].view(dtype).view(L, 2, T + 1, C_)[:, :, T].contiguous().view(torch.uint8)
    want = ref[:g.n].view(dtype).view(L, 2, T + 1, C_)[:, :, T].contiguous().view(torch.uint8)
    assert torch.equal(spare, want), "a spare row between the planes was written"
    g.check(what="serving cache")


def test_step_functions_write_nothing_past_their_outputs(cg, synth_mod):
    from kv_cache_compression_cg_gb300 import capi
    lib = capi.load()
    k, v, Tc, bk, bv = _case(synth_mod, "ragged")
    L, T, C_ = k.shape
    kt, vt = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    shp = cg.make_shape(L, T, C_, Tc)
    bk_a, bv_a = np.asarray(bk, np.int32), np.asarray(bv, np.int32)
    pk, pv = C.c_void_p(bk_a.ctypes.data), C.c_void_p(bv_a.ctypes.data)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: C.c_void_p(t.data_ptr())
    ns = 2 * L * T
    st = Guarded(4, torch.int32)
    st.t.zero_()
    sym = Guarded(2 * L * T * C_)
    max1 = Guarded(4 * L * T, torch.int16)
    assert lib.cg_quantize(p(kt), p(vt), C.byref(shp), pk, pv, p(sym.t), p(max1.t), p(st.t), stream) == 0
    ncdf = int(lib.cg_cdf_elems(C.byref(shp), pk, pv))
    cdf = Guarded(2 * ncdf, torch.int16)
    assert lib.cg_calculate_cdf(p(sym.t), C.byref(shp), pk, pv, p(cdf.t), p(st.t), stream) == 0
    cap = int(lib.cg_max_compressed_bytes(C.byref(shp)))
    wsb = int(lib.cg_workspace_bytes(C.byref(shp)))
    ws = Guarded(wsb)
    packed = Guarded(cap)
    ln = Guarded(4 * ns, torch.int32)
    off = Guarded(8 * (ns + 1), torch.int64)
    assert lib.cg_encode(p(sym.t), p(cdf.t), C.byref(shp), pk, pv, p(packed.t), cap, p(ln.t), p(off.t), p(ws.t),
                         wsb, p(st.t), stream) == 0
    sym2 = Guarded(2 * L * T * C_)
    assert lib.cg_decode(p(packed.t), cap, p(off.t), p(ln.t), p(cdf.t), C.byref(shp), pk, pv, p(sym2.t), p(st.t),
                         stream) == 0
    out_k, out_v = Guarded(4 * L * T * C_, torch.float32), Guarded(4 * L * T * C_, torch.float32)
    assert lib.cg_dequantize(p(sym2.t), p(max1.t), C.byref(shp), pk, pv, p(out_k.t), p(out_v.t), p(st.t),
                             stream) == 0
    dsym = Guarded(2 * L * T * C_)
    dmax1 = Guarded(4 * L * T, torch.int16)
    assert lib.cg_quantize_delta(p(kt), p(vt), C.byref(shp), pk, pv, 5, p(dsym.t), p(dmax1.t), p(st.t),
                                 stream) == 0
    dk, dv = Guarded(4 * L * T * C_, torch.float32), Guarded(4 * L * T * C_, torch.float32)
    assert lib.cg_dequantize_delta(p(dsym.t), p(dmax1.t), C.byref(shp), pk, pv, 5, p(dk.t), p(dv.t), p(st.t),
                                   stream) == 0
    torch.cuda.synchronize()
    assert int(st.t.item()) == 0
    assert torch.equal(sym2.t, sym.t)
    total = int(off.t[-1].item())
    packed.check(total, "cg_encode packed past off[nstreams]")
    for what, gg in (("sym", sym), ("max1", max1), ("cdf", cdf), ("workspace", ws), ("len", ln), ("off", off),
                     ("decoded sym", sym2), ("out_k", out_k), ("out_v", out_v), ("delta sym", dsym),
                     ("delta max1", dmax1), ("delta out_k", dk), ("delta out_v", dv), ("status", st)):
        gg.check(what=what)


def test_noalloc_writes_nothing_past_its_outputs(cg, synth_mod):
    from kv_cache_compression_cg_gb300 import capi
    lib = capi.load()
    w = synth_mod.WORKLOADS["tiny"]
    k, v = synth_mod.generate(w)
    kt, vt = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    shp = cg.make_shape(w.L, w.T, w.C, w.chunk_tokens)
    bk_a, bv_a = np.asarray(w.bins_k, np.int32), np.asarray(w.bins_v, np.int32)
    pk, pv = C.c_void_p(bk_a.ctypes.data), C.c_void_p(bv_a.ctypes.data)
    p = lambda t: C.c_void_p(t.data_ptr())
    ns = 2 * w.L * w.T
    cap = int(lib.cg_max_compressed_bytes(C.byref(shp)))
    max1 = Guarded(4 * w.L * w.T, torch.int16)
    cdf = Guarded(2 * int(lib.cg_cdf_elems(C.byref(shp), pk, pv)), torch.int16)
    packed = Guarded(cap)
    ln = Guarded(4 * ns, torch.int32)
    off = Guarded(8 * (ns + 1), torch.int64)
    st = Guarded(4, torch.int32)
    st.t.zero_()
    rc = lib.cg_compress_chunk_noalloc(p(kt), p(vt), C.byref(shp), pk, pv, p(max1.t), p(cdf.t), p(packed.t), cap,
                                       p(ln.t), p(off.t), p(st.t),
                                       C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.t.item()) == 0
    packed.check(int(off.t[-1].item()), "packed past off[nstreams]")
    for what, gg in (("max1", max1), ("cdf", cdf), ("len", ln), ("off", off), ("status", st)):
        gg.check(what=what)
