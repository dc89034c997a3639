"""CPU oracle for the CacheGen KV-cache codec (ctypes wrapper over cg_oracle.c).

TEST INFRASTRUCTURE ONLY. The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers. The product library
(``kv_cache_compression_cg_gb300``) never imports this package and has no CPU
fallback.

Citation key: [CG] is the web page "CacheGen 技术详解：KV Cache 的高效压缩与流式传输"
(CacheGen as implemented in LMCache). The arithmetic lives in cg_oracle.c;
this module only moves numpy arrays across the C boundary.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cg_oracle.c")
_SO = os.path.join(_HERE, "libcg_oracle.so")
_LOCK = threading.Lock()
_LIB = None

OK, ERR_ARG, ERR_NONFINITE, ERR_CAPACITY, ERR_CORRUPT, ERR_NOMEM = range(6)


def build(force: bool = False) -> str:
    """Compile cg_oracle.c with gcc (plain C11, no fused multiply-add)."""
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "cg_oracle.h")))
    if force or stale:
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
             "-fPIC", "-shared", "-Wall", "-Wextra", _SRC, "-o", tmp, "-lm"],
            check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> C.CDLL:
    global _LIB
    with _LOCK:
        if _LIB is None:
            build()
            L = C.CDLL(_SO)
            p = C.c_void_p
            i32, i64, u64 = C.c_int32, C.c_int64, C.c_uint64
            sig = {
                "orc_half_to_float": (C.c_float, [C.c_uint16]),
                "orc_quantize_group": (C.c_int, [p, i64, C.c_int, p, p]),
                "orc_dequantize_value": (C.c_float, [C.c_uint8, C.c_int, C.c_uint16]),
                "orc_cdf_from_counts": (C.c_int, [p, C.c_int, C.c_uint32, p]),
                "orc_encode_stream": (i64, [p, i64, p, i64, C.c_int, p, i64]),
                "orc_decode_stream": (C.c_int, [p, i64, i64, p, i64, C.c_int, p, p]),
                "orc_num_streams": (i64, [C.c_int, C.c_int]),
                "orc_cdf_elems": (i64, [C.c_int] * 6),
                "orc_cdf_offset": (i64, [C.c_int] * 8),
                "orc_stream_id": (i64, [C.c_int] * 7),
                "orc_alphabet": (C.c_int, [p, C.c_int]),
                "orc_quantize": (C.c_int, [p, p, C.c_int, C.c_int, C.c_int, i64, p, p, p, p]),
                "orc_calculate_cdf": (C.c_int, [p, C.c_int, C.c_int, C.c_int, C.c_int,
                                                C.c_int, C.c_int, p]),
                "orc_encode": (C.c_int, [p, p] + [C.c_int] * 6 + [p, u64, p, p]),
                "orc_decode": (C.c_int, [p, p, p, p] + [C.c_int] * 6 + [p]),
                "orc_dequantize": (C.c_int, [p, p, C.c_int, C.c_int, C.c_int, p, p, p, p]),
                "orc_compress": (C.c_int, [p, p, C.c_int, C.c_int, C.c_int, C.c_int, i64,
                                           p, p, p, p, p, u64, p, p]),
                "orc_decompress": (C.c_int, [p, p, p, p, p] + [C.c_int] * 4 + [p, p, p, p]),
                "orc_alphabet_v2": (C.c_int, [C.c_int]),
                "orc_float_to_half": (C.c_uint16, [C.c_float]),
                "orc_dequantize_half": (C.c_int, [p, p, C.c_int, C.c_int, C.c_int, p, p, p, p]),
                "orc_rec_bytes": (i64, [C.c_int] * 4 + [p, p]),
                "orc_rec_offset": (i64, [C.c_int, C.c_int, p, p] + [C.c_int] * 4),
                "orc_record_from_counts": (C.c_int, [p, C.c_int, p]),
                "orc_counts_from_record": (C.c_int, [p, C.c_int, C.c_uint32, p]),
                "orc_cdf_from_counts_mode": (C.c_int, [p, C.c_int, C.c_uint32, C.c_int, p]),
                "orc_compress_v2": (C.c_int, [p, p, C.c_int, C.c_int, C.c_int, C.c_int, i64,
                                              p, p, p, p, p, u64, p, p]),
                "orc_decompress_v2": (C.c_int, [p, p, p, p, p] + [C.c_int] * 4 + [p, p, p, p]),
                "orc_v3_fixed_bytes": (i64, [C.c_int] * 4),
                "orc_v3_max_bytes": (i64, [C.c_int] * 4 + [p, p]),
                "orc_records_to_v3": (i64, [p] + [C.c_int] * 4 + [p, p, p, i64]),
                "orc_v3_to_records": (C.c_int, [p, i64] + [C.c_int] * 4 + [p, p, p]),
                "orc_compress_v3": (C.c_int, [p, p] + [C.c_int] * 5 + [i64, p, p, p, p, i64, p, p, u64, p, p]),
                "orc_decompress_v3": (C.c_int, [p, p, p, i64, p] + [C.c_int] * 5 + [p, p, p, p]),
                "orc_half_up": (C.c_uint16, [C.c_float]),
                "orc_floats_to_half": (None, [p, i64, p]),
                "orc_quantize_delta": (C.c_int, [p, p] + [C.c_int] * 5 + [i64, p, p, p, p]),
                "orc_dequantize_delta": (C.c_int, [p, p] + [C.c_int] * 5 + [p, p, p, p]),
                "orc_compress_ex": (C.c_int, [p, p] + [C.c_int] * 6 + [i64, p, p, p, p, p, u64, p, p]),
                "orc_decompress_ex": (C.c_int, [p, p, p, p, p] + [C.c_int] * 6 + [p, p, p, p]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _ = i32
            _LIB = L
    return _LIB


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code}")
        self.code = code


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return C.c_void_p(a.ctypes.data)


def _check(code: int, what: str):
    if code != OK:
        raise OracleError(code, what)


def _bits(x: np.ndarray) -> np.ndarray:
    """fp16 array (or its uint16 bits) -> contiguous uint16 bits."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    assert x.dtype == np.uint16
    return x


def _bins(b, L) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(b, dtype=np.int32))
    assert b.shape == (L,)
    return b


# ----------------------------------------------------------------------------
# single-group / single-stream primitives
# ----------------------------------------------------------------------------
def half_to_float(h: int) -> float:
    return lib().orc_half_to_float(int(h))


def quantize_group(x, bins: int):
    """[CG §2.3(1)] one group -> (uint8 symbols, max1 as fp16 bits)."""
    x = _bits(np.asarray(x))
    q = np.empty(x.size, np.uint8)
    m = np.zeros(1, np.uint16)
    _check(lib().orc_quantize_group(_ptr(x), x.size, int(bins), _ptr(q), _ptr(m)),
           "quantize_group")
    return q, int(m[0])


def dequantize_value(q: int, bins: int, max1_bits: int) -> float:
    """[CG §2.4(2)] one symbol -> binary32 value (returned as a Python float)."""
    return lib().orc_dequantize_value(int(q), int(bins), int(max1_bits))


def cdf_from_counts(n, Tk: int | None = None) -> np.ndarray:
    """[CG §2.3(2)] counts -> uint16 CDF entries cdf[0..A-1]."""
    n = np.ascontiguousarray(np.asarray(n, dtype=np.uint32))
    Tk = int(n.sum()) if Tk is None else int(Tk)
    out = np.empty(n.size, np.uint16)
    _check(lib().orc_cdf_from_counts(_ptr(n), n.size, Tk, _ptr(out)), "cdf_from_counts")
    return out


def encode_stream(sym, cdf_rows: np.ndarray) -> bytes:
    """Encode sym[i] with CDF row cdf_rows[i] (shape [n, A], or [A] for all)."""
    sym = np.ascontiguousarray(np.asarray(sym, dtype=np.uint8))
    rows = np.ascontiguousarray(np.asarray(cdf_rows, dtype=np.uint16))
    A = rows.shape[-1]
    stride = A if rows.ndim == 2 else 0
    if rows.ndim == 2:
        assert rows.shape[0] == sym.size
    cap = 2 * sym.size + 8
    out = np.zeros(cap, np.uint8)
    n = lib().orc_encode_stream(_ptr(sym), sym.size, _ptr(rows), stride, A, _ptr(out), cap)
    if n < 0:
        raise OracleError(ERR_ARG, "encode_stream")
    return out[:n].tobytes()


def decode_stream(data: bytes, n: int, cdf_rows: np.ndarray):
    """Decode n symbols; returns (symbols, bytes consumed, status)."""
    buf = np.frombuffer(bytes(data) + b"\0", np.uint8)  # never a zero-size pointer
    rows = np.ascontiguousarray(np.asarray(cdf_rows, dtype=np.uint16))
    A = rows.shape[-1]
    stride = A if rows.ndim == 2 else 0
    sym = np.zeros(max(n, 1), np.uint8)
    used = np.zeros(1, np.int64)
    st = lib().orc_decode_stream(_ptr(buf), len(data), n, _ptr(rows), stride, A,
                                 _ptr(sym), _ptr(used))
    return sym[:n], int(used[0]), st


# ----------------------------------------------------------------------------
# layout helpers
# ----------------------------------------------------------------------------
def alphabet(bins) -> int:
    b = np.ascontiguousarray(np.asarray(bins, dtype=np.int32))
    return lib().orc_alphabet(_ptr(b), b.size)


def num_streams(L: int, T: int) -> int:
    return lib().orc_num_streams(L, T)


def cdf_elems(L, T, C_, Tc, A_k, A_v) -> int:
    return lib().orc_cdf_elems(L, T, C_, Tc, A_k, A_v)


def cdf_offset(L, C_, A_k, A_v, k, kv, l, c) -> int:
    return lib().orc_cdf_offset(L, C_, A_k, A_v, k, kv, l, c)


def stream_id(L, T, Tc, k, kv, l, tl) -> int:
    return lib().orc_stream_id(L, T, Tc, k, kv, l, tl)


# ----------------------------------------------------------------------------
# whole-tensor steps
# ----------------------------------------------------------------------------
def quantize(k, v, bins_k, bins_v=None):
    """k, v: fp16 [L][T][C] -> (sym uint8 [2][L][T][C], max1 fp16 bits [2][L][T])."""
    k, v = _bits(k), _bits(v)
    L, T, C_ = k.shape
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    sym = np.empty((2, L, T, C_), np.uint8)
    max1 = np.empty((2, L, T), np.uint16)
    _check(lib().orc_quantize(_ptr(k), _ptr(v), L, T, C_, T * C_, _ptr(bk), _ptr(bv),
                              _ptr(sym), _ptr(max1)), "quantize")
    return sym, max1


def calculate_cdf(sym, Tc: int, A_k: int, A_v: int) -> np.ndarray:
    sym = np.ascontiguousarray(sym, dtype=np.uint8)
    _, L, T, C_ = sym.shape
    cdf = np.empty(cdf_elems(L, T, C_, Tc, A_k, A_v), np.uint16)
    _check(lib().orc_calculate_cdf(_ptr(sym), L, T, C_, Tc, A_k, A_v, _ptr(cdf)),
           "calculate_cdf")
    return cdf


def max_compressed_bytes(L: int, T: int, C_: int) -> int:
    return num_streams(L, T) * (2 * C_ + 8)


def encode(sym, cdf, Tc: int, A_k: int, A_v: int, capacity: int | None = None):
    sym = np.ascontiguousarray(sym, dtype=np.uint8)
    _, L, T, C_ = sym.shape
    cdf = np.ascontiguousarray(cdf, dtype=np.uint16)
    ns = num_streams(L, T)
    cap = max_compressed_bytes(L, T, C_) if capacity is None else int(capacity)
    packed = np.zeros(max(cap, 1), np.uint8)
    ln = np.empty(ns, np.uint32)
    off = np.empty(ns + 1, np.uint64)
    st = lib().orc_encode(_ptr(sym), _ptr(cdf), L, T, C_, Tc, A_k, A_v, _ptr(packed),
                          cap, _ptr(ln), _ptr(off))
    if st not in (OK, ERR_CAPACITY):
        raise OracleError(st, "encode")
    total = int(off[-1])
    return packed[:min(total, cap)].copy(), ln, off, st


def decode(packed, off, ln, cdf, L, T, C_, Tc, A_k, A_v):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    if packed.size == 0:
        packed = np.zeros(1, np.uint8)
    sym = np.empty((2, L, T, C_), np.uint8)
    st = lib().orc_decode(_ptr(packed), _ptr(np.ascontiguousarray(off, np.uint64)),
                          _ptr(np.ascontiguousarray(ln, np.uint32)),
                          _ptr(np.ascontiguousarray(cdf, np.uint16)),
                          L, T, C_, Tc, A_k, A_v, _ptr(sym))
    return sym, st


def dequantize(sym, max1, bins_k, bins_v=None):
    sym = np.ascontiguousarray(sym, dtype=np.uint8)
    _, L, T, C_ = sym.shape
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    out_k = np.empty((L, T, C_), np.float32)
    out_v = np.empty((L, T, C_), np.float32)
    _check(lib().orc_dequantize(_ptr(sym), _ptr(np.ascontiguousarray(max1, np.uint16)),
                                L, T, C_, _ptr(bk), _ptr(bv), _ptr(out_k), _ptr(out_v)),
           "dequantize")
    return out_k, out_v


def compress(k, v, Tc: int, bins_k, bins_v=None):
    """Quantise -> CDF -> encode. Returns a dict with max1, cdf, packed, len, off."""
    k, v = _bits(k), _bits(v)
    L, T, C_ = k.shape
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    A_k, A_v = alphabet(bk), alphabet(bv)
    ns = num_streams(L, T)
    cap = max_compressed_bytes(L, T, C_)
    max1 = np.empty((2, L, T), np.uint16)
    cdf = np.empty(cdf_elems(L, T, C_, Tc, A_k, A_v), np.uint16)
    packed = np.zeros(cap, np.uint8)
    ln = np.empty(ns, np.uint32)
    off = np.empty(ns + 1, np.uint64)
    _check(lib().orc_compress(_ptr(k), _ptr(v), L, T, C_, Tc, T * C_, _ptr(bk), _ptr(bv),
                              _ptr(max1), _ptr(cdf), _ptr(packed), cap, _ptr(ln), _ptr(off)),
           "compress")
    return {"max1": max1, "cdf": cdf, "packed": packed[:int(off[-1])].copy(),
            "len": ln, "off": off, "A_k": A_k, "A_v": A_v}


def decompress(packed, off, ln, cdf, max1, L, T, C_, Tc, bins_k, bins_v=None):
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    if packed.size == 0:
        packed = np.zeros(1, np.uint8)
    out_k = np.empty((L, T, C_), np.float32)
    out_v = np.empty((L, T, C_), np.float32)
    _check(lib().orc_decompress(_ptr(packed), _ptr(np.ascontiguousarray(off, np.uint64)),
                                _ptr(np.ascontiguousarray(ln, np.uint32)),
                                _ptr(np.ascontiguousarray(cdf, np.uint16)),
                                _ptr(np.ascontiguousarray(max1, np.uint16)),
                                L, T, C_, Tc, _ptr(bk), _ptr(bv), _ptr(out_k), _ptr(out_v)),
           "decompress")
    return out_k, out_v


# ----------------------------------------------------------------------------
# format 2: side information as symbol counts
# ----------------------------------------------------------------------------
def alphabet_v2(bins: int) -> int:
    """A = 2*MAX + 1 symbols for a layer with `bins` bins."""
    return lib().orc_alphabet_v2(int(bins))


def rec_bytes(L, T, C_, Tc, bins_k, bins_v=None) -> int:
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    return int(lib().orc_rec_bytes(L, T, C_, Tc, _ptr(bk), _ptr(bv)))


def rec_offset(L, C_, bins_k, bins_v, k, kv, l, c) -> int:
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    return int(lib().orc_rec_offset(L, C_, _ptr(bk), _ptr(bv), k, kv, l, c))


def record_from_counts(counts) -> np.ndarray:
    n = np.ascontiguousarray(np.asarray(counts, dtype=np.uint32))
    rec = np.zeros(n.size, np.uint8)
    _check(lib().orc_record_from_counts(_ptr(n), n.size, _ptr(rec)), "record_from_counts")
    return rec


def counts_from_record(rec, Tk: int) -> np.ndarray:
    r = np.ascontiguousarray(np.asarray(rec, dtype=np.uint8))
    n = np.zeros(r.size, np.uint32)
    _check(lib().orc_counts_from_record(_ptr(r), r.size, int(Tk), _ptr(n)), "counts_from_record")
    return n


def cdf_from_counts_mode(counts, Tk: int, mode: int) -> np.ndarray:
    n = np.ascontiguousarray(np.asarray(counts, dtype=np.uint32))
    cdf = np.zeros(n.size, np.uint16)
    _check(lib().orc_cdf_from_counts_mode(_ptr(n), n.size, int(Tk), int(mode), _ptr(cdf)),
           "cdf_from_counts_mode")
    return cdf


def compress_v2(k, v, Tc: int, bins_k, bins_v=None):
    """Format 2: quantise -> counts -> records -> encode. Returns max1, rec,
    packed, len, off."""
    k, v = _bits(k), _bits(v)
    L, T, C_ = k.shape
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    ns = num_streams(L, T)
    cap = max_compressed_bytes(L, T, C_)
    max1 = np.empty((2, L, T), np.uint16)
    rec = np.zeros(max(rec_bytes(L, T, C_, Tc, bk, bv), 1), np.uint8)
    packed = np.zeros(max(cap, 1), np.uint8)
    ln = np.empty(max(ns, 1), np.uint32)
    off = np.empty(ns + 1, np.uint64)
    _check(lib().orc_compress_v2(_ptr(k), _ptr(v), L, T, C_, Tc, T * C_, _ptr(bk), _ptr(bv),
                                 _ptr(max1), _ptr(rec), _ptr(packed), cap, _ptr(ln), _ptr(off)),
           "compress_v2")
    nrec = rec_bytes(L, T, C_, Tc, bk, bv)
    return {"max1": max1, "rec": rec[:nrec].copy(), "packed": packed[:int(off[-1])].copy(),
            "len": ln[:ns], "off": off}


def decompress_v2(packed, off, ln, rec, max1, L, T, C_, Tc, bins_k, bins_v=None):
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    if packed.size == 0:
        packed = np.zeros(1, np.uint8)
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    if rec.size == 0:
        rec = np.zeros(1, np.uint8)
    out_k = np.empty((L, T, C_), np.float32)
    out_v = np.empty((L, T, C_), np.float32)
    _check(lib().orc_decompress_v2(_ptr(packed), _ptr(np.ascontiguousarray(off, np.uint64)),
                                   _ptr(np.ascontiguousarray(ln, np.uint32)), _ptr(rec),
                                   _ptr(np.ascontiguousarray(max1, np.uint16)),
                                   L, T, C_, Tc, _ptr(bk), _ptr(bv), _ptr(out_k), _ptr(out_v)),
           "decompress_v2")
    return out_k, out_v


# ----------------------------------------------------------------------------
# serving layouts: binary16 output
# ----------------------------------------------------------------------------
def float_to_half(x: float) -> int:
    """binary32 -> binary16 bits, round to nearest, ties to even."""
    return int(lib().orc_float_to_half(float(np.float32(x))))


def dequantize_half(sym, max1, bins_k, bins_v=None):
    """sym [2][L][T][C] + max1 [2][L][T] -> binary16 K, V [L][T][C] (as uint16 bits)."""
    sym = np.ascontiguousarray(sym, dtype=np.uint8)
    _, L, T, C_ = sym.shape
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    out_k = np.empty((L, T, C_), np.uint16)
    out_v = np.empty((L, T, C_), np.uint16)
    _check(lib().orc_dequantize_half(_ptr(sym), _ptr(np.ascontiguousarray(max1, np.uint16)), L, T, C_,
                                     _ptr(bk), _ptr(bv), _ptr(out_k), _ptr(out_v)), "dequantize_half")
    return out_k, out_v


# ----------------------------------------------------------------------------
# token-locality delta (specification G)
# ----------------------------------------------------------------------------
def half_up(m: float) -> int:
    """The smallest binary16 value >= m, as bits (65504's bits above it)."""
    return int(lib().orc_half_up(float(np.float32(m))))


def floats_to_half(x) -> np.ndarray:
    """binary32 array -> binary16 bits (uint16), round to nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_floats_to_half(_ptr(x), x.size, _ptr(out))
    return out


def quantize_delta(k, v, Tc: int, G: int, bins_k, bins_v=None):
    """QA + QD: symbols [2][L][T][C] and max1 [2][L][T] (fp16 bits)."""
    k, v = _bits(k), _bits(v)
    L, T, C_ = k.shape
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    sym = np.empty((2, L, T, C_), np.uint8)
    max1 = np.empty((2, L, T), np.uint16)
    _check(lib().orc_quantize_delta(_ptr(k), _ptr(v), L, T, C_, Tc, G, T * C_, _ptr(bk), _ptr(bv),
                                    _ptr(sym), _ptr(max1)), "quantize_delta")
    return sym, max1


def dequantize_delta(sym, max1, Tc: int, G: int, bins_k, bins_v=None):
    """D on anchors, DD elsewhere: binary32 K, V [L][T][C]."""
    sym = np.ascontiguousarray(sym, dtype=np.uint8)
    _, L, T, C_ = sym.shape
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    out_k = np.empty((L, T, C_), np.float32)
    out_v = np.empty((L, T, C_), np.float32)
    _check(lib().orc_dequantize_delta(_ptr(sym), _ptr(np.ascontiguousarray(max1, np.uint16)), L, T, C_,
                                      Tc, G, _ptr(bk), _ptr(bv), _ptr(out_k), _ptr(out_v)),
           "dequantize_delta")
    return out_k, out_v


def compress_ex(k, v, Tc: int, bins_k, bins_v=None, fmt: int = 1, group: int = 1):
    """Quantise with token groups of `group` (1: plain) and code in format
    `fmt`. Returns max1, side ("cdf" or "rec"), packed, len, off."""
    k, v = _bits(k), _bits(v)
    L, T, C_ = k.shape
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    ns = num_streams(L, T)
    cap = max_compressed_bytes(L, T, C_)
    max1 = np.empty((2, L, T), np.uint16)
    if fmt == 1:
        side = np.empty(max(cdf_elems(L, T, C_, Tc, alphabet(bk), alphabet(bv)), 1), np.uint16)
    else:
        side = np.zeros(max(rec_bytes(L, T, C_, Tc, bk, bv), 1), np.uint8)
    packed = np.zeros(max(cap, 1), np.uint8)
    ln = np.empty(max(ns, 1), np.uint32)
    off = np.empty(ns + 1, np.uint64)
    _check(lib().orc_compress_ex(_ptr(k), _ptr(v), L, T, C_, Tc, group, fmt, T * C_, _ptr(bk), _ptr(bv),
                                 _ptr(max1), _ptr(side), _ptr(packed), cap, _ptr(ln), _ptr(off)),
           "compress_ex")
    n_side = cdf_elems(L, T, C_, Tc, alphabet(bk), alphabet(bv)) if fmt == 1 else rec_bytes(L, T, C_, Tc, bk, bv)
    return {"max1": max1, "cdf" if fmt == 1 else "rec": side[:n_side].copy(),
            "packed": packed[:int(off[-1])].copy(), "len": ln[:ns], "off": off}


def decompress_ex(packed, off, ln, side, max1, L, T, C_, Tc, bins_k, bins_v=None, fmt: int = 1,
                  group: int = 1):
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    if packed.size == 0:
        packed = np.zeros(1, np.uint8)
    side = np.ascontiguousarray(side, dtype=np.uint16 if fmt == 1 else np.uint8)
    if side.size == 0:
        side = np.zeros(1, side.dtype)
    out_k = np.empty((L, T, C_), np.float32)
    out_v = np.empty((L, T, C_), np.float32)
    _check(lib().orc_decompress_ex(_ptr(packed), _ptr(np.ascontiguousarray(off, np.uint64)),
                                   _ptr(np.ascontiguousarray(ln, np.uint32)), _ptr(side),
                                   _ptr(np.ascontiguousarray(max1, np.uint16)),
                                   L, T, C_, Tc, group, fmt, _ptr(bk), _ptr(bv), _ptr(out_k), _ptr(out_v)),
           "decompress_ex")
    return out_k, out_v


# ----------------------------------------------------------------------------
# format 3: compact count records
# ----------------------------------------------------------------------------
def v3_fixed_bytes(L, T, C_, Tc) -> int:
    return int(lib().orc_v3_fixed_bytes(L, T, C_, Tc))


def v3_max_bytes(L, T, C_, Tc, bins_k, bins_v=None) -> int:
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    return int(lib().orc_v3_max_bytes(L, T, C_, Tc, _ptr(bk), _ptr(bv)))


def records_to_v3(rec, L, T, C_, Tc, bins_k, bins_v=None) -> np.ndarray:
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    cap = v3_max_bytes(L, T, C_, Tc, bk, bv)
    side = np.zeros(max(cap, 1), np.uint8)
    n = lib().orc_records_to_v3(_ptr(np.ascontiguousarray(rec, np.uint8)), L, T, C_, Tc, _ptr(bk), _ptr(bv),
                                _ptr(side), cap)
    if n < 0:
        raise OracleError(int(-n), "records_to_v3")
    return side[:n].copy()


def v3_to_records(side, L, T, C_, Tc, bins_k, bins_v=None) -> np.ndarray:
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    side = np.ascontiguousarray(side, np.uint8)
    rec = np.zeros(max(rec_bytes(L, T, C_, Tc, bk, bv), 1), np.uint8)
    _check(lib().orc_v3_to_records(_ptr(side if side.size else np.zeros(1, np.uint8)), side.size, L, T, C_, Tc,
                                   _ptr(bk), _ptr(bv), _ptr(rec)), "v3_to_records")
    return rec[:rec_bytes(L, T, C_, Tc, bk, bv)]


def compress_v3(k, v, Tc: int, bins_k, bins_v=None, group: int = 1):
    """Format 3: returns max1, side (the whole side buffer), packed, len, off."""
    k, v = _bits(k), _bits(v)
    L, T, C_ = k.shape
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    ns = num_streams(L, T)
    cap = max_compressed_bytes(L, T, C_)
    scap = v3_max_bytes(L, T, C_, Tc, bk, bv)
    max1 = np.empty((2, L, T), np.uint16)
    side = np.zeros(max(scap, 1), np.uint8)
    nside = np.zeros(1, np.int64)
    packed = np.zeros(max(cap, 1), np.uint8)
    ln = np.empty(max(ns, 1), np.uint32)
    off = np.empty(ns + 1, np.uint64)
    _check(lib().orc_compress_v3(_ptr(k), _ptr(v), L, T, C_, Tc, group, T * C_, _ptr(bk), _ptr(bv), _ptr(max1),
                                 _ptr(side), scap, _ptr(nside), _ptr(packed), cap, _ptr(ln), _ptr(off)),
           "compress_v3")
    return {"max1": max1, "side": side[:int(nside[0])].copy(), "packed": packed[:int(off[-1])].copy(),
            "len": ln[:ns], "off": off}


def decompress_v3(packed, ln, side, max1, L, T, C_, Tc, bins_k, bins_v=None, group: int = 1):
    bk = _bins(bins_k, L)
    bv = _bins(bins_k if bins_v is None else bins_v, L)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    if packed.size == 0:
        packed = np.zeros(1, np.uint8)
    side = np.ascontiguousarray(side, np.uint8)
    out_k = np.empty((L, T, C_), np.float32)
    out_v = np.empty((L, T, C_), np.float32)
    _check(lib().orc_decompress_v3(_ptr(packed), _ptr(np.ascontiguousarray(ln, np.uint32)), _ptr(side), side.size,
                                   _ptr(np.ascontiguousarray(max1, np.uint16)), L, T, C_, Tc, group, _ptr(bk),
                                   _ptr(bv), _ptr(out_k), _ptr(out_v)), "decompress_v3")
    return out_k, out_v
