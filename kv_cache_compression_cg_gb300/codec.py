"""PyTorch-facing wrappers of the C ABI: PyTorch only provides device memory
and the current stream; every computation runs in libcachegen_gb300.so.

Tensors crossing the boundary: fp16 K and V [L][T][C] (any layer stride),
uint16 data (max1 bits, CDF entries) carried in torch.int16 storage, uint32
lengths in torch.int32, uint64 offsets in torch.int64.
"""
from __future__ import annotations

import ctypes as C
import dataclasses

import numpy as np
import torch

from . import capi

__all__ = ["Codec", "Compressed", "quantize", "calculate_cdf", "encode", "decode", "dequantize",
           "quantize_delta", "dequantize_delta", "compress_chunk", "decompress_chunk", "make_shape"]


def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream: torch.cuda.Stream | None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _bins(b, L: int) -> np.ndarray:
    arr = np.ascontiguousarray(np.asarray(b, dtype=np.int32))
    if arr.shape != (L,):
        raise ValueError(f"bins must have {L} entries, got shape {arr.shape}")
    return arr


def _np_ptr(a: np.ndarray | None):
    return None if a is None else C.c_void_p(a.ctypes.data)


def make_shape(L: int, T: int, C_: int, chunk_tokens: int = 256,
               layer_stride: int | None = None) -> capi.cg_shape:
    return capi.cg_shape(L, T, C_, chunk_tokens, T * C_ if layer_stride is None else layer_stride)


def _kv_shape(k: torch.Tensor, v: torch.Tensor, chunk_tokens: int) -> capi.cg_shape:
    if k.dtype != torch.float16 or v.dtype != torch.float16:
        raise TypeError("K and V must be torch.float16")
    if not (k.is_cuda and v.is_cuda):
        raise ValueError("K and V must be CUDA tensors")
    if k.dim() != 3 or k.shape != v.shape:
        raise ValueError("K and V must both be [L, T, C]")
    L, T, C_ = k.shape
    if k.stride(2) != 1 or k.stride(1) != C_ or v.stride() != k.stride():
        raise ValueError("K and V need contiguous [T, C] planes with equal layer strides")
    return make_shape(L, T, C_, chunk_tokens, k.stride(0))


@dataclasses.dataclass
class Compressed:
    """Device-resident output of compress: the serialised form of a chunk."""
    L: int
    T: int
    C: int
    chunk_tokens: int
    bins_k: np.ndarray
    bins_v: np.ndarray
    max1: torch.Tensor      # int16 [2, L, T] (fp16 bits)
    cdf: torch.Tensor       # int16 [cdf_elems] (uint16 entries)
    packed: torch.Tensor    # uint8 [capacity]
    len: torch.Tensor       # int32 [nstreams] (uint32)
    off: torch.Tensor       # int64 [nstreams + 1]
    status: torch.Tensor    # int32 [1]
    fmt: int = 1            # 1: CDF entries in `cdf`; 2: count records in `rec`
    rec: torch.Tensor | None = None  # uint8 [record bytes] (format 2)
    group: int = 1          # token-locality delta group (1: none)
    side3: torch.Tensor | None = None  # uint8 [capacity] (format 3 side buffer)
    side3_fixed: int = 0    # format 3: bytes before the counts (offV)

    def side3_bytes(self) -> int:
        """Format 3: the side buffer's size, offV + O[nslice]."""
        ns = 2 * self.L * (-(-self.T // self.chunk_tokens))
        vbytes = int(self.side3[8 * ns:8 * ns + 8].cpu().numpy().view(np.uint64)[0])
        return self.side3_fixed + vbytes

    @property
    def shape(self) -> capi.cg_shape:
        return make_shape(self.L, self.T, self.C, self.chunk_tokens)

    def total_bytes(self) -> int:
        return int(self.off[-1].item())


class Codec:
    """Pre-allocated buffers for repeated compress/decompress of one shape.

    The C library allocates nothing; this object owns every buffer (outputs,
    workspace, status word) so a timed loop allocates nothing either.
    """

    def __init__(self, L: int, T: int, C_: int, bins_k, bins_v=None, chunk_tokens: int = 256,
                 capacity: int | None = None, device: str | torch.device = "cuda", fmt: int = 1,
                 group: int = 1):
        """fmt: 1 (CDF entries), 2 (count records) or 3 (compact count
        records; offsets rebuilt from the lengths); group: token-locality
        delta group size [CG §1.2(1)] (1: no delta; > 1 needs chunk_tokens
        <= 256 to decode)."""
        if fmt not in (1, 2, 3):
            raise ValueError("fmt must be 1 (CDF entries), 2 (count records) or 3 (compact records)")
        if not 1 <= group <= 1024:
            raise ValueError("group must be in [1, 1024]")
        if group > 1 and chunk_tokens > 256:
            raise ValueError("the delta decodes only chunks of at most 256 tokens")
        self.fmt = fmt
        self.group = group
        self.L, self.T, self.C, self.chunk_tokens = L, T, C_, chunk_tokens
        self.bins_k = _bins(bins_k, L)
        self.bins_v = _bins(bins_k if bins_v is None else bins_v, L)
        lib = capi.load()
        shp = make_shape(L, T, C_, chunk_tokens)
        self.nstreams = int(lib.cg_num_streams(C.byref(shp)))
        self.cdf_elems = int(lib.cg_cdf_elems(C.byref(shp), _np_ptr(self.bins_k), _np_ptr(self.bins_v)))
        self.rec_bytes = int(lib.cg_record_bytes(C.byref(shp), _np_ptr(self.bins_k), _np_ptr(self.bins_v)))
        if fmt >= 2 and self.rec_bytes == 0 and T > 0:
            raise ValueError("formats 2 and 3 need chunk_tokens <= 256")
        self.side3_cap = int(lib.cg_side3_max_bytes(C.byref(shp), _np_ptr(self.bins_k), _np_ptr(self.bins_v)))
        if fmt == 3 and self.side3_cap == 0 and T > 0:
            raise ValueError("format 3 needs every layer alphabet within 32 symbols")
        self.max_bytes = int(lib.cg_max_compressed_bytes(C.byref(shp)))
        if self.nstreams == 0 and T > 0 or self.cdf_elems == 0 and T > 0:
            raise ValueError("invalid shape or bins for the codec")
        self.capacity = self.max_bytes if capacity is None else int(capacity)
        self.ws_bytes = int(lib.cg_compress_workspace_bytes(C.byref(shp)))
        if fmt == 3:
            self.ws_bytes = max(self.ws_bytes, int(lib.cg_workspace_bytes_v3(
                C.byref(shp), _np_ptr(self.bins_k), _np_ptr(self.bins_v))))
        dev = torch.device(device)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.out = Compressed(
            L, T, C_, chunk_tokens, self.bins_k, self.bins_v,
            max1=torch.empty((2, L, T), dtype=torch.int16, device=dev),
            cdf=torch.empty(max(self.cdf_elems if fmt == 1 else 1, 1), dtype=torch.int16, device=dev),
            packed=torch.empty(max(self.capacity, 16), dtype=torch.uint8, device=dev),
            len=torch.empty(max(self.nstreams, 1), dtype=torch.int32, device=dev),
            off=torch.empty(self.nstreams + 1, dtype=torch.int64, device=dev),
            status=torch.zeros(1, dtype=torch.int32, device=dev), fmt=fmt,
            rec=torch.empty(max(self.rec_bytes, 1), dtype=torch.uint8, device=dev) if fmt == 2 else None,
            group=group,
            side3=torch.empty(max(self.side3_cap, 8), dtype=torch.uint8, device=dev) if fmt == 3 else None,
            side3_fixed=int(lib.cg_side3_fixed_bytes(C.byref(shp))) if fmt == 3 else 0)
        self.out_k = torch.empty((L, T, C_), dtype=torch.float32, device=dev)
        self.out_v = torch.empty((L, T, C_), dtype=torch.float32, device=dev)
        self.dstatus = torch.zeros(1, dtype=torch.int32, device=dev)

    def compress(self, k: torch.Tensor, v: torch.Tensor, stream=None) -> Compressed:
        shp = _kv_shape(k, v, self.chunk_tokens)
        if (shp.L, shp.T, shp.C) != (self.L, self.T, self.C):
            raise ValueError("K/V shape differs from the codec's")
        o = self.out
        if self.fmt == 3:
            capi.check(capi.load().cg_compress_chunk_v3(
                _ptr(k), _ptr(v), C.byref(shp), _np_ptr(self.bins_k), _np_ptr(self.bins_v), self.group,
                _ptr(o.max1), _ptr(o.side3), self.side3_cap, _ptr(o.packed), self.capacity, _ptr(o.len), _ptr(o.off),
                _ptr(self.workspace), self.ws_bytes, _ptr(o.status), _stream(stream)), "cg_compress_chunk_v3")
            return o
        if self.group > 1:
            capi.check(capi.load().cg_compress_chunk_ex(
                _ptr(k), _ptr(v), C.byref(shp), _np_ptr(self.bins_k), _np_ptr(self.bins_v), self.fmt, self.group,
                _ptr(o.max1), _ptr(o.cdf if self.fmt == 1 else o.rec), _ptr(o.packed), self.capacity, _ptr(o.len),
                _ptr(o.off), _ptr(self.workspace), self.ws_bytes, _ptr(o.status), _stream(stream)),
                "cg_compress_chunk_ex")
            return o
        if self.fmt == 2:
            capi.check(capi.load().cg_compress_chunk_v2(
                _ptr(k), _ptr(v), C.byref(shp), _np_ptr(self.bins_k), _np_ptr(self.bins_v),
                _ptr(o.max1), _ptr(o.rec), _ptr(o.packed), self.capacity, _ptr(o.len), _ptr(o.off),
                _ptr(self.workspace), self.ws_bytes, _ptr(o.status), _stream(stream)),
                "cg_compress_chunk_v2")
            return o
        capi.check(capi.load().cg_compress_chunk(
            _ptr(k), _ptr(v), C.byref(shp), _np_ptr(self.bins_k), _np_ptr(self.bins_v),
            _ptr(o.max1), _ptr(o.cdf), _ptr(o.packed), self.capacity, _ptr(o.len), _ptr(o.off),
            _ptr(self.workspace), self.ws_bytes, _ptr(o.status), _stream(stream)),
            "cg_compress_chunk")
        return o

    def decompress(self, c: Compressed | None = None, stream=None):
        c = self.out if c is None else c
        shp = make_shape(c.L, c.T, c.C, c.chunk_tokens)
        if c.group > 1 or c.fmt == 3:
            self.decompress_into(self.out_k, self.out_v, c, stream)
            return self.out_k, self.out_v
        if c.fmt == 2:
            capi.check(capi.load().cg_decompress_chunk_v2(
                _ptr(c.packed), c.packed.numel(), _ptr(c.off), _ptr(c.len), _ptr(c.rec), _ptr(c.max1),
                C.byref(shp), _np_ptr(c.bins_k), _np_ptr(c.bins_v), _ptr(self.out_k), _ptr(self.out_v),
                _ptr(self.dstatus), _stream(stream)), "cg_decompress_chunk_v2")
            return self.out_k, self.out_v
        capi.check(capi.load().cg_decompress_chunk(
            _ptr(c.packed), c.packed.numel(), _ptr(c.off), _ptr(c.len), _ptr(c.cdf), _ptr(c.max1),
            C.byref(shp), _np_ptr(c.bins_k), _np_ptr(c.bins_v), _ptr(self.out_k), _ptr(self.out_v),
            _ptr(self.dstatus), _stream(stream)), "cg_decompress_chunk")
        return self.out_k, self.out_v


    def decompress_into(self, out_k: torch.Tensor, out_v: torch.Tensor, c: Compressed | None = None,
                        stream=None) -> None:
        """Decompress straight into a serving layout: out_k / out_v are
        float32 or float16 [L, T, C] views with contiguous [T, C] planes and
        the same layer stride (e.g. buf[:, 0] and buf[:, 1] of a [L, 2, T, C]
        cache). float16 gets each binary32 value rounded to nearest-even."""
        c = self.out if c is None else c
        if out_k.dtype != out_v.dtype or out_k.dtype not in (torch.float32, torch.float16):
            raise TypeError("outputs must both be float32 or both float16")
        if tuple(out_k.shape) != (c.L, c.T, c.C) or out_v.shape != out_k.shape:
            raise ValueError("outputs must be [L, T, C]")
        if out_k.stride(2) != 1 or out_k.stride(1) != c.C or out_v.stride() != out_k.stride():
            raise ValueError("outputs need contiguous [T, C] planes with equal layer strides")
        shp = make_shape(c.L, c.T, c.C, c.chunk_tokens)
        if c.fmt == 3:
            capi.check(capi.load().cg_decompress_chunk_v3(
                _ptr(c.packed), c.packed.numel(), _ptr(c.len), _ptr(c.side3), c.side3.numel(), _ptr(c.max1),
                C.byref(shp), _np_ptr(c.bins_k), _np_ptr(c.bins_v), c.group,
                capi.CG_OUT_F16 if out_k.dtype == torch.float16 else capi.CG_OUT_F32,
                _ptr(out_k), _ptr(out_v), out_k.stride(0), _ptr(self.workspace), self.ws_bytes,
                _ptr(self.dstatus), _stream(stream)), "cg_decompress_chunk_v3")
            return
        side = c.cdf if c.fmt == 1 else c.rec
        capi.check(capi.load().cg_decompress_chunk_ex(
            _ptr(c.packed), c.packed.numel(), _ptr(c.off), _ptr(c.len), _ptr(side), _ptr(c.max1),
            C.byref(shp), _np_ptr(c.bins_k), _np_ptr(c.bins_v), c.fmt, c.group,
            capi.CG_OUT_F16 if out_k.dtype == torch.float16 else capi.CG_OUT_F32,
            _ptr(out_k), _ptr(out_v), out_k.stride(0), _ptr(self.dstatus), _stream(stream)),
            "cg_decompress_chunk_ex")


# ---------------------------------------------------------------------------
# one-shot step functions (allocate their outputs with torch)
# ---------------------------------------------------------------------------
def quantize(k, v, bins_k, bins_v=None, chunk_tokens: int = 256, status=None, stream=None):
    """[CG §2.3(1)] -> (sym uint8 [2, L, T, C], max1 int16 [2, L, T])."""
    shp = _kv_shape(k, v, chunk_tokens)
    bk = _bins(bins_k, shp.L)
    bv = _bins(bins_k if bins_v is None else bins_v, shp.L)
    sym = torch.empty((2, shp.L, shp.T, shp.C), dtype=torch.uint8, device=k.device)
    max1 = torch.empty((2, shp.L, shp.T), dtype=torch.int16, device=k.device)
    capi.check(capi.load().cg_quantize(_ptr(k), _ptr(v), C.byref(shp), _np_ptr(bk), _np_ptr(bv),
                                       _ptr(sym), _ptr(max1), _ptr(status), _stream(stream)),
               "cg_quantize")
    return sym, max1


def calculate_cdf(sym, bins_k, bins_v=None, chunk_tokens: int = 256, status=None, stream=None):
    """[CG §2.3(2)] symbols [2, L, T, C] -> CDF entries (int16 storage)."""
    _, L, T, C_ = sym.shape
    shp = make_shape(L, T, C_, chunk_tokens)
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    n = int(capi.load().cg_cdf_elems(C.byref(shp), _np_ptr(bk), _np_ptr(bv)))
    cdf = torch.empty(max(n, 1), dtype=torch.int16, device=sym.device)
    capi.check(capi.load().cg_calculate_cdf(_ptr(sym), C.byref(shp), _np_ptr(bk), _np_ptr(bv),
                                            _ptr(cdf), _ptr(status), _stream(stream)),
               "cg_calculate_cdf")
    return cdf


def encode(sym, cdf, bins_k, bins_v=None, chunk_tokens: int = 256, capacity: int | None = None,
           status=None, stream=None):
    """[CG §1.2(3)] -> (packed uint8, len int32, off int64)."""
    _, L, T, C_ = sym.shape
    shp = make_shape(L, T, C_, chunk_tokens)
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    lib = capi.load()
    ns = int(lib.cg_num_streams(C.byref(shp)))
    cap = int(lib.cg_max_compressed_bytes(C.byref(shp))) if capacity is None else int(capacity)
    wsb = int(lib.cg_workspace_bytes(C.byref(shp)))
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=sym.device)
    packed = torch.empty(max(cap, 16), dtype=torch.uint8, device=sym.device)
    ln = torch.empty(max(ns, 1), dtype=torch.int32, device=sym.device)
    off = torch.empty(ns + 1, dtype=torch.int64, device=sym.device)
    capi.check(lib.cg_encode(_ptr(sym), _ptr(cdf), C.byref(shp), _np_ptr(bk), _np_ptr(bv),
                             _ptr(packed), cap, _ptr(ln), _ptr(off), _ptr(ws), wsb, _ptr(status),
                             _stream(stream)), "cg_encode")
    return packed, ln, off


def decode(packed, off, ln, cdf, L, T, C_, bins_k, bins_v=None, chunk_tokens: int = 256,
           status=None, stream=None, packed_bytes: int | None = None):
    """[CG §2.4(1)] -> sym uint8 [2, L, T, C]."""
    shp = make_shape(L, T, C_, chunk_tokens)
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    sym = torch.empty((2, L, T, C_), dtype=torch.uint8, device=packed.device)
    nbytes = packed.numel() if packed_bytes is None else int(packed_bytes)
    capi.check(capi.load().cg_decode(_ptr(packed), nbytes, _ptr(off), _ptr(ln), _ptr(cdf),
                                     C.byref(shp), _np_ptr(bk), _np_ptr(bv), _ptr(sym),
                                     _ptr(status), _stream(stream)), "cg_decode")
    return sym


def dequantize(sym, max1, bins_k, bins_v=None, chunk_tokens: int = 256, stream=None):
    """[CG §2.4(2)] -> (out_k, out_v) float32 [L, T, C]."""
    _, L, T, C_ = sym.shape
    shp = make_shape(L, T, C_, chunk_tokens)
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    ok = torch.empty((L, T, C_), dtype=torch.float32, device=sym.device)
    ov = torch.empty((L, T, C_), dtype=torch.float32, device=sym.device)
    capi.check(capi.load().cg_dequantize(_ptr(sym), _ptr(max1), C.byref(shp), _np_ptr(bk),
                                         _np_ptr(bv), _ptr(ok), _ptr(ov), None, _stream(stream)),
               "cg_dequantize")
    return ok, ov


def quantize_delta(k, v, group: int, bins_k, bins_v=None, chunk_tokens: int = 256, status=None,
                   stream=None):
    """[CG §1.2(1)] anchors + deltas per token group -> (sym, max1) as quantize."""
    shp = _kv_shape(k, v, chunk_tokens)
    bk = _bins(bins_k, shp.L)
    bv = _bins(bins_k if bins_v is None else bins_v, shp.L)
    sym = torch.empty((2, shp.L, shp.T, shp.C), dtype=torch.uint8, device=k.device)
    max1 = torch.empty((2, shp.L, shp.T), dtype=torch.int16, device=k.device)
    capi.check(capi.load().cg_quantize_delta(_ptr(k), _ptr(v), C.byref(shp), _np_ptr(bk), _np_ptr(bv), group,
                                             _ptr(sym), _ptr(max1), _ptr(status), _stream(stream)),
               "cg_quantize_delta")
    return sym, max1


def dequantize_delta(sym, max1, group: int, bins_k, bins_v=None, chunk_tokens: int = 256, stream=None):
    """The inverse of quantize_delta's symbols -> (out_k, out_v) float32 [L, T, C]."""
    _, L, T, C_ = sym.shape
    shp = make_shape(L, T, C_, chunk_tokens)
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    ok = torch.empty((L, T, C_), dtype=torch.float32, device=sym.device)
    ov = torch.empty((L, T, C_), dtype=torch.float32, device=sym.device)
    capi.check(capi.load().cg_dequantize_delta(_ptr(sym), _ptr(max1), C.byref(shp), _np_ptr(bk), _np_ptr(bv),
                                               group, _ptr(ok), _ptr(ov), None, _stream(stream)),
               "cg_dequantize_delta")
    return ok, ov


def compress_chunk(k, v, bins_k, bins_v=None, chunk_tokens: int = 256,
                   capacity: int | None = None, stream=None) -> Compressed:
    """Quantise -> CDF -> encode -> pack (one call into the library)."""
    L, T, C_ = k.shape
    codec = Codec(L, T, C_, bins_k, bins_v, chunk_tokens, capacity, device=k.device)
    return codec.compress(k, v, stream)


def decompress_chunk(c: Compressed, stream=None):
    """Decode fused with dequantisation -> (out_k, out_v) float32."""
    codec = _DecodeOnly(c)
    return codec.run(stream)


class _DecodeOnly:
    def __init__(self, c: Compressed):
        self.c = c
        dev = c.packed.device
        self.out_k = torch.empty((c.L, c.T, c.C), dtype=torch.float32, device=dev)
        self.out_v = torch.empty((c.L, c.T, c.C), dtype=torch.float32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def run(self, stream=None):
        c = self.c
        shp = make_shape(c.L, c.T, c.C, c.chunk_tokens)
        capi.check(capi.load().cg_decompress_chunk(
            _ptr(c.packed), c.packed.numel(), _ptr(c.off), _ptr(c.len), _ptr(c.cdf), _ptr(c.max1),
            C.byref(shp), _np_ptr(c.bins_k), _np_ptr(c.bins_v), _ptr(self.out_k), _ptr(self.out_v),
            _ptr(self.status), _stream(stream)), "cg_decompress_chunk")
        return self.out_k, self.out_v
