"""ctypes binding of include/cachegen.h (same function names, argument
marshalling only). Every step runs in the CUDA library; there is no Python or
CPU fallback: if the library is missing this module raises on first use."""
from __future__ import annotations

import ctypes as C
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcachegen_gb300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "cachegen.h")

CG_OK, CG_ERR_INVALID_ARG, CG_ERR_WORKSPACE, CG_ERR_CUDA = 0, 1, 2, 3
CG_FLAG_NONFINITE, CG_FLAG_CAPACITY, CG_FLAG_CORRUPT, CG_FLAG_BAD_SYMBOL = 0x1, 0x2, 0x4, 0x8
CG_FLAG_TIMEOUT = 0x10
CG_MAX_LAYERS, CG_MAX_CHUNK_TOKENS, CG_MAX_CHANNELS = 1024, 1024, 65536
CG_NOALLOC_WORKSPACE_BYTES = 64 << 20
CG_OUT_F32, CG_OUT_F16 = 0, 1

_ERRORS = {CG_ERR_INVALID_ARG: "invalid argument", CG_ERR_WORKSPACE: "workspace too small",
           CG_ERR_CUDA: "CUDA launch failed"}


class cg_shape(C.Structure):
    _fields_ = [("L", C.c_int32), ("T", C.c_int32), ("C", C.c_int32),
                ("chunk_tokens", C.c_int32), ("layer_stride", C.c_int64)]


class CodecError(RuntimeError):
    def __init__(self, code: int, fn: str):
        super().__init__(f"{fn}: {_ERRORS.get(code, 'error')} (cg_status {code})")
        self.code = code


_p, _u64, _i32 = C.c_void_p, C.c_uint64, C.c_int32
_SHAPE = C.POINTER(cg_shape)
SIGNATURES = {
    "cg_num_streams": (_u64, [_SHAPE]),
    "cg_cdf_elems": (_u64, [_SHAPE, _p, _p]),
    "cg_max_compressed_bytes": (_u64, [_SHAPE]),
    "cg_workspace_bytes": (_u64, [_SHAPE]),
    "cg_compress_workspace_bytes": (_u64, [_SHAPE]),
    "cg_quantize": (_i32, [_p, _p, _SHAPE, _p, _p, _p, _p, _p, _p]),
    "cg_calculate_cdf": (_i32, [_p, _SHAPE, _p, _p, _p, _p, _p]),
    "cg_encode": (_i32, [_p, _p, _SHAPE, _p, _p, _p, _u64, _p, _p, _p, _u64, _p, _p]),
    "cg_decode": (_i32, [_p, _u64, _p, _p, _p, _SHAPE, _p, _p, _p, _p, _p]),
    "cg_dequantize": (_i32, [_p, _p, _SHAPE, _p, _p, _p, _p, _p, _p]),
    "cg_compress_chunk": (_i32, [_p, _p, _SHAPE, _p, _p, _p, _p, _p, _u64, _p, _p, _p, _u64,
                                 _p, _p]),
    "cg_decompress_chunk": (_i32, [_p, _u64, _p, _p, _p, _p, _SHAPE, _p, _p, _p, _p, _p, _p]),
    "cg_compress_chunk_noalloc": (_i32, [_p, _p, _SHAPE, _p, _p, _p, _p, _p, _u64, _p, _p, _p, _p]),
    "cg_record_bytes": (_u64, [_SHAPE, _p, _p]),
    "cg_compress_chunk_v2": (_i32, [_p, _p, _SHAPE, _p, _p, _p, _p, _p, _u64, _p, _p, _p, _u64,
                                    _p, _p]),
    "cg_decompress_chunk_v2": (_i32, [_p, _u64, _p, _p, _p, _p, _SHAPE, _p, _p, _p, _p, _p, _p]),
    "cg_decompress_chunk_ex": (_i32, [_p, _u64, _p, _p, _p, _p, _SHAPE, _p, _p, C.c_int, C.c_int32, C.c_int,
                                      _p, _p, C.c_int64, _p, _p]),
    "cg_quantize_delta": (_i32, [_p, _p, _SHAPE, _p, _p, C.c_int32, _p, _p, _p, _p]),
    "cg_side3_fixed_bytes": (_u64, [_SHAPE]),
    "cg_side3_max_bytes": (_u64, [_SHAPE, _p, _p]),
    "cg_workspace_bytes_v3": (_u64, [_SHAPE, _p, _p]),
    "cg_compress_chunk_v3": (_i32, [_p, _p, _SHAPE, _p, _p, C.c_int32, _p, _p, _u64, _p, _u64, _p, _p, _p, _u64,
                                    _p, _p]),
    "cg_decompress_chunk_v3": (_i32, [_p, _u64, _p, _p, _u64, _p, _SHAPE, _p, _p, C.c_int32, C.c_int, _p, _p,
                                      C.c_int64, _p, _u64, _p, _p]),
    "cg_dequantize_delta": (_i32, [_p, _p, _SHAPE, _p, _p, C.c_int32, _p, _p, _p, _p]),
    "cg_compress_chunk_ex": (_i32, [_p, _p, _SHAPE, _p, _p, C.c_int, C.c_int32, _p, _p, _p, _u64, _p, _p, _p,
                                    _u64, _p, _p]),
    "cg_version": (C.c_char_p, []),
}

_LOCK = threading.Lock()
_LIB = None


def header_functions() -> list[str]:
    """Names of the functions include/cachegen.h declares."""
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cg_[a-z0-9_]+)\s*\(", text)))


def load() -> C.CDLL:
    """Load libcachegen_gb300.so (built by kv_cache_compression_cg_gb300.build)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA codec library missing at {LIB_PATH}; build it with "
                    "`python -m kv_cache_compression_cg_gb300.build` (no CPU fallback exists)")
            lib = C.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = lib
    return _LIB


def check(code: int, fn: str) -> None:
    if code != CG_OK:
        raise CodecError(code, fn)


def __getattr__(name):
    if name in SIGNATURES:
        return getattr(load(), name)
    raise AttributeError(name)
