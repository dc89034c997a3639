"""Seeded synthetic KV-cache inputs (fp16 K and V of shape [L][T][C]).

The generator (synth.c) holds none of the codec's arithmetic; it serves the
CUDA tests, the oracle tests and the benchmark alike, so all of them see the
same bytes. Model KV caches need trained weights and prompts, which are not
available, so these seeded tensors stand in for them, with the shapes and
value statistics of the workloads below.

Workloads (per K and per V):
  tiny          [2, 64, 64]        one chunk of 64; bins 32 (layer 0), 16 (layer 1);
                                   AR(1) rho=0.9, sigma_c ~ LogNormal(0, 0.5); seed 0
  mistral_chunk [32, 256, 1024]    one chunk; bins 32 for layers 0-9, 16 for 10-31;
                                   AR(1) rho=0.9, LogNormal(0, 0.5), 2% outlier
                                   channels at x8; seed 1
  ctx4096       [32, 4096, 1024]   16 chunks of 256; as mistral_chunk; seed 2
  ctx32k        [48, 32768, 1024]  128 chunks; bins 32 for layers 0-15, 16 for
                                   16-47; AR(1) rho=0.95, LogNormal(0, 0.7), 2% x8;
                                   seed 3
  stress80k     [32, 81920, 1024]  320 chunks; bins 8 everywhere; i.i.d.
                                   Student-t(3) x sigma_c, LogNormal(0, 0.5); seed 4
  uniform       [32, 256, 1024]    one chunk; bins as mistral_chunk; U[0, 1)
                                   (the CacheGen page's torch.rand check); seed 5
"""
from __future__ import annotations

import ctypes as C
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libcg_synth.so")
_LOCK = threading.Lock()
_LIB = None

AR1, STUDENT_T, UNIFORM = 0, 1, 2


class _Params(C.Structure):
    _fields_ = [("kind", C.c_int32), ("L", C.c_int32), ("T", C.c_int32), ("C", C.c_int32),
                ("seed", C.c_uint64), ("rho", C.c_double), ("sigma_log", C.c_double),
                ("outlier_frac", C.c_double), ("outlier_scale", C.c_double)]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int
    T: int
    C: int
    chunk_tokens: int
    bins_k: tuple
    bins_v: tuple
    kind: int
    seed: int
    rho: float = 0.0
    sigma_log: float = 0.5
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0

    @property
    def n_chunks(self) -> int:
        return -(-self.T // self.chunk_tokens)

    @property
    def elements(self) -> int:
        return 2 * self.L * self.T * self.C

    def params(self, L=None, T=None, C_=None) -> _Params:
        return _Params(self.kind, L or self.L, T or self.T, C_ or self.C, self.seed,
                       self.rho, self.sigma_log, self.outlier_frac, self.outlier_scale)

    def describe(self) -> str:
        kinds = {AR1: f"AR(1) rho={self.rho}", STUDENT_T: "iid Student-t(3)",
                 UNIFORM: "U[0,1)"}
        out = (f", {self.outlier_frac:.0%} outlier channels x{self.outlier_scale:g}"
               if self.outlier_frac else "")
        sig = "" if self.kind == UNIFORM else f", sigma_c~LogNormal(0,{self.sigma_log})"
        return (f"{self.name}: K,V fp16 [{self.L},{self.T},{self.C}], "
                f"{self.n_chunks} chunk(s) of {self.chunk_tokens}, "
                f"{kinds[self.kind]}{sig}{out}, seed {self.seed}")


def _split_bins(L, boundary, hi, lo):
    return tuple([hi] * boundary + [lo] * (L - boundary))


WORKLOADS = {
    "tiny": Workload("tiny", 2, 64, 64, 64, (32, 16), (32, 16), AR1, 0, rho=0.9),
    "mistral_chunk": Workload("mistral_chunk", 32, 256, 1024, 256, _split_bins(32, 10, 32, 16),
                              _split_bins(32, 10, 32, 16), AR1, 1, rho=0.9,
                              outlier_frac=0.02, outlier_scale=8.0),
    "ctx4096": Workload("ctx4096", 32, 4096, 1024, 256, _split_bins(32, 10, 32, 16),
                        _split_bins(32, 10, 32, 16), AR1, 2, rho=0.9,
                        outlier_frac=0.02, outlier_scale=8.0),
    "ctx32k": Workload("ctx32k", 48, 32768, 1024, 256, _split_bins(48, 16, 32, 16),
                       _split_bins(48, 16, 32, 16), AR1, 3, rho=0.95, sigma_log=0.7,
                       outlier_frac=0.02, outlier_scale=8.0),
    "stress80k": Workload("stress80k", 32, 81920, 1024, 256, (8,) * 32, (8,) * 32,
                          STUDENT_T, 4),
    "uniform": Workload("uniform", 32, 256, 1024, 256, _split_bins(32, 10, 32, 16),
                        _split_bins(32, 10, 32, 16), UNIFORM, 5),
}


_CORE = os.path.join(_HERE, "synth_core.h")
_GPU_SRC = os.path.join(_HERE, "synth_gpu.cu")
_GPU_SO = os.path.join(_HERE, "libcg_synth_gpu.so")
_GPU_LIB = None


def build(force: bool = False) -> str:
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < max(
        os.path.getmtime(_SRC), os.path.getmtime(_CORE))
    if force or stale:
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                        "-fPIC", "-shared", "-pthread", "-Wall", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> C.CDLL:
    global _LIB
    with _LOCK:
        if _LIB is None:
            build()
            L = C.CDLL(_SO)
            L.syn_generate.restype = C.c_int
            L.syn_generate.argtypes = [C.POINTER(_Params), C.c_void_p, C.c_void_p,
                                       C.c_int64, C.c_int]
            L.syn_generate_slice_range.restype = C.c_int
            L.syn_generate_slice_range.argtypes = [C.POINTER(_Params), C.c_int, C.c_int, C.c_int,
                                                   C.c_int, C.c_void_p]
            L.syn_slice_sigma.restype = C.c_int
            L.syn_slice_sigma.argtypes = [C.POINTER(_Params), C.c_int, C.c_int, C.c_void_p]
            L.syn_generate_slice.restype = C.c_int
            L.syn_generate_slice.argtypes = [C.POINTER(_Params), C.c_int, C.c_int,
                                             C.c_void_p]
            L.syn_ln.restype = C.c_double
            L.syn_ln.argtypes = [C.c_double]
            L.syn_expo.restype = C.c_double
            L.syn_expo.argtypes = [C.c_double]
            L.syn_cis2pi.restype = None
            L.syn_cis2pi.argtypes = [C.c_double, C.POINTER(C.c_double), C.POINTER(C.c_double)]
            L.syn_half.restype = C.c_uint16
            L.syn_half.argtypes = [C.c_double]
            L.syn_splitmix.restype = C.c_uint64
            L.syn_splitmix.argtypes = [C.c_uint64, C.c_uint64]
            _LIB = L
    return _LIB


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def generate_into(w: Workload, k_ptr: int, v_ptr: int, layer_stride: int | None = None,
                  T: int | None = None, nthreads: int | None = None) -> None:
    """Fill caller-owned host memory (e.g. pinned tensors) with K and V."""
    p = w.params(T=T)
    ls = (T or w.T) * w.C if layer_stride is None else layer_stride
    rc = lib().syn_generate(C.byref(p), C.c_void_p(k_ptr), C.c_void_p(v_ptr), ls,
                            nthreads or _threads())
    if rc != 0:
        raise RuntimeError("synthetic generator failed")


def generate(w: Workload | str, T: int | None = None, nthreads: int | None = None):
    """Return (k, v) as numpy float16 arrays [L][T][C].

    ``T`` overrides the token count (the first T tokens of the same seeded
    sequence; AR(1) state is carried along tokens, so a prefix is identical to
    the prefix of the full tensor)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    Tn = T or w.T
    k = np.empty((w.L, Tn, w.C), np.float16)
    v = np.empty((w.L, Tn, w.C), np.float16)
    generate_into(w, k.ctypes.data, v.ctypes.data, T=Tn, nthreads=nthreads)
    return k, v


def generate_slice(w: Workload | str, kv: int, layer: int, T: int | None = None) -> np.ndarray:
    """One (kv, layer) slice [T][C] as float16, generated alone."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    Tn = T or w.T
    out = np.empty((Tn, w.C), np.float16)
    p = w.params(T=Tn)
    if lib().syn_generate_slice(C.byref(p), kv, layer, C.c_void_p(out.ctypes.data)) != 0:
        raise RuntimeError("synthetic generator failed")
    return out


def generate_slice_range(w: Workload | str, kv: int, layer: int, t0: int, t1: int) -> np.ndarray:
    """Tokens [t0, t1) of one (kv, layer) slice, [t1 - t0][C] float16."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    out = np.empty((t1 - t0, w.C), np.float16)
    p = w.params(T=max(t1, 1))
    if lib().syn_generate_slice_range(C.byref(p), kv, layer, t0, t1, C.c_void_p(out.ctypes.data)) != 0:
        raise RuntimeError("synthetic generator failed")
    return out


def sigmas(w: Workload) -> np.ndarray:
    """Per-channel sigma_c of every slice, float64 [2][L][C]."""
    out = np.zeros((2, w.L, w.C), np.float64)
    if w.kind == UNIFORM:
        return out
    p = w.params()
    for kv in range(2):
        for layer in range(w.L):
            if lib().syn_slice_sigma(C.byref(p), kv, layer, C.c_void_p(out[kv, layer].ctypes.data)) != 0:
                raise RuntimeError("synthetic generator failed")
    return out


# ---------------------------------------------------------------------------
# device generator (same bytes as the host one, for the full-size workloads)
# ---------------------------------------------------------------------------
def build_device(force: bool = False) -> str:
    stale = (not os.path.exists(_GPU_SO)) or os.path.getmtime(_GPU_SO) < max(
        os.path.getmtime(_GPU_SRC), os.path.getmtime(_CORE))
    if force or stale:
        import shutil
        nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
        tmp = _GPU_SO + f".{os.getpid()}.tmp"
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false",
                        "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared", _GPU_SRC, "-o", tmp],
                       check=True)
        os.replace(tmp, _GPU_SO)
    return _GPU_SO


def _gpu_lib() -> C.CDLL:
    global _GPU_LIB
    with _LOCK:
        if _GPU_LIB is None:
            build_device()
            L = C.CDLL(_GPU_SO)
            L.syn_generate_device.restype = C.c_int
            L.syn_generate_device.argtypes = [C.POINTER(_Params), C.c_void_p, C.c_void_p, C.c_void_p,
                                              C.c_int64, C.c_void_p]
            _GPU_LIB = L
    return _GPU_LIB


def generate_device(w: Workload | str, T: int | None = None, device="cuda"):
    """K and V as torch float16 CUDA tensors [L][T][C], generated on the
    device with the host generator's arithmetic (identical bytes)."""
    import torch
    if isinstance(w, str):
        w = WORKLOADS[w]
    Tn = T or w.T
    lib()  # host library (sigmas)
    k = torch.empty((w.L, Tn, w.C), dtype=torch.float16, device=device)
    v = torch.empty((w.L, Tn, w.C), dtype=torch.float16, device=device)
    sig = torch.from_numpy(sigmas(w).reshape(-1)).to(device)
    p = w.params(T=Tn)
    stream = torch.cuda.current_stream(k.device).cuda_stream
    rc = _gpu_lib().syn_generate_device(C.byref(p), C.c_void_p(sig.data_ptr()), C.c_void_p(k.data_ptr()),
                                        C.c_void_p(v.data_ptr()), Tn * w.C, C.c_void_p(stream))
    if rc != 0:
        raise RuntimeError("device generator launch failed")
    torch.cuda.current_stream(k.device).synchronize()
    return k, v
