"""Chunk-pipelined streaming between pinned host memory and the GPU.

The page streams a context's KV cache chunk by chunk: chunks are coded
independently, so a chunk can be sent while the next one is still being
encoded ([CG §1.2(4)], chunk-wise processing; [CG §2.3(2)], one CDF set per
chunk). `StreamingCodec` does that on one GPU with six CUDA streams:

- sender: the fp16 K, V rows of piece p (a run of whole chunks) go host to
  device on the copy-in stream while piece p - 1 is compressed on the coding
  stream; each compressed piece goes back to pinned host buffers on the
  copy-out stream as soon as it is done;
- receiver: each host piece is copied in and decompressed as soon as its bytes
  are on the host, while later pieces are still moving.

A piece's compressed bytes are exactly the bytes of those chunks in a
whole-tensor call (streams are chunk-major), so `shard.assemble` of the pieces'
host arrays gives the whole tensor's compressed form. Every coding step runs in
the CUDA library through `codec.Codec`; this module only orders copies and
launches.
"""
from __future__ import annotations

import ctypes as C
import ctypes.util
import dataclasses
import os

import numpy as np
import torch

from . import codec as _codec

__all__ = ["StreamingCodec", "HostPiece", "AdaptiveLevels"]

_MEMCPY_H2D = 1
_rt = None


def _cudart():
    """The CUDA runtime, for strided (2D) asynchronous copies."""
    global _rt
    if _rt is None:
        cands = [ctypes.util.find_library("cudart"), "/usr/local/cuda/lib64/libcudart.so"]
        for c in cands:
            if c and (os.path.exists(c) or not os.path.isabs(c)):
                try:
                    lib = C.CDLL(c)
                    break
                except OSError:
                    continue
        else:
            raise RuntimeError("CUDA runtime library not found")
        lib.cudaMemcpy2DAsync.restype = C.c_int
        lib.cudaMemcpy2DAsync.argtypes = [C.c_void_p, C.c_size_t, C.c_void_p, C.c_size_t, C.c_size_t,
                                          C.c_size_t, C.c_int, C.c_void_p]
        lib.cudaMemcpyAsync.restype = C.c_int
        lib.cudaMemcpyAsync.argtypes = [C.c_void_p, C.c_void_p, C.c_size_t, C.c_int, C.c_void_p]
        _rt = lib
    return _rt


_MEMCPY_DEFAULT = 4  # direction from the pointers (unified addressing)


def _copy(dst: torch.Tensor, src: torch.Tensor, nbytes: int, stream: torch.cuda.Stream):
    """Asynchronous copy of the first nbytes of src to dst on `stream` (one
    runtime call; torch's copy_ between pinned host and device memory spends
    a few hundred microseconds on the host, which would stall the pipeline)."""
    if nbytes <= 0:
        return
    if nbytes > dst.numel() * dst.element_size() or nbytes > src.numel() * src.element_size():
        raise ValueError("copy larger than a buffer")
    err = _cudart().cudaMemcpyAsync(C.c_void_p(dst.data_ptr()), C.c_void_p(src.data_ptr()), nbytes,
                                    _MEMCPY_DEFAULT, C.c_void_p(stream.cuda_stream))
    if err != 0:
        raise RuntimeError(f"cudaMemcpyAsync failed ({err})")


def _nb(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


@dataclasses.dataclass
class HostPiece:
    """Compressed tokens [t0, t1) in pinned host memory (one codec call)."""
    t0: int
    t1: int
    nbytes: int
    packed: torch.Tensor   # uint8 [capacity]; bytes [0, nbytes) are the streams
    len: torch.Tensor      # int32 [2 L (t1 - t0)] (uint32)
    off: torch.Tensor      # int64 [2 L (t1 - t0) + 1]
    side: torch.Tensor     # format 1: int16 CDF entries; 2: uint8 count records; 3: uint8 side buffer
    max1: torch.Tensor     # int16 [2, L, t1 - t0] (fp16 bits)
    ready: torch.cuda.Event
    fmt: int = 1
    side_bytes: int = 0    # format 3: the side buffer's size (the rest of `side` is unused)
    level: int = 0         # index of the bins this piece was quantised with

    def arrays(self) -> dict:
        """numpy views in the layout `shard.assemble` joins (formats 1, 2)."""
        side = ("cdf", self.side.numpy().view(np.uint16)) if self.fmt == 1 else ("rec", self.side.numpy())
        return {"max1": self.max1.numpy().view(np.uint16), side[0]: side[1],
                "packed": self.packed[:self.nbytes].numpy(), "len": self.len.numpy().view(np.uint32),
                "off": self.off.numpy().view(np.uint64)}


class AdaptiveLevels:
    """Bandwidth-adaptive choice of the quantisation level per piece: chunks
    are small so the coder can follow a changing link [CG §2.3(3)]. Levels are
    ordered finest first (most bins); a piece gets the finest level whose
    compressed size, estimated from the pieces already sent at that level
    (bytes per token, averaged with weight `smoothing` on the newest), fits
    the link's rate times the time budget of a piece. A level not yet seen is
    taken as fitting (so it gets measured); with nothing fitting, the
    coarsest. Host logic only: the rate is the caller's measurement of its
    link."""

    def __init__(self, nlevels: int, seconds_per_piece: float, bytes_per_second: float,
                 smoothing: float = 0.5, prior_bytes_per_token=None):
        if nlevels < 1 or seconds_per_piece <= 0 or bytes_per_second <= 0 or not 0 < smoothing <= 1:
            raise ValueError("need nlevels >= 1, positive budget and rate, smoothing in (0, 1]")
        self.n = nlevels
        self.seconds = seconds_per_piece
        self.rate = bytes_per_second
        self.smoothing = smoothing
        self.est = list(prior_bytes_per_token) if prior_bytes_per_token is not None else [None] * nlevels
        if len(self.est) != nlevels:
            raise ValueError("one prior per level")

    def set_rate(self, bytes_per_second: float):
        if bytes_per_second <= 0:
            raise ValueError("the rate must be positive")
        self.rate = bytes_per_second

    def level_for(self, tokens: int) -> int:
        budget = self.rate * self.seconds
        for lv in range(self.n):
            e = self.est[lv]
            if e is None or e * tokens <= budget:
                return lv
        return self.n - 1

    def observe(self, level: int, tokens: int, nbytes: int):
        per = nbytes / max(tokens, 1)
        e = self.est[level]
        self.est[level] = per if e is None else (1 - self.smoothing) * e + self.smoothing * per


class StreamingCodec:
    """Pipelined compress from pinned host K, V and decompress of host pieces.

    All buffers (device staging of the fp16 input, one sender and one receiver
    codec per piece and quantisation level, pinned host pieces) are allocated
    once here.
    """

    def __init__(self, L: int, T: int, C_: int, bins_k, bins_v=None, chunk_tokens: int = 256,
                 piece_chunks: int = 2, device: str | torch.device = "cuda", fmt: int = 1, group: int = 1,
                 levels=None):
        """fmt, group: the codec's format and token-locality delta group (as
        Codec); pieces are whole chunks, so they code independently. levels:
        optional list of (bins_k, bins_v), finest first, that pieces may
        switch between (`stream_pieces(policy=...)`); default the one pair."""
        if piece_chunks < 1:
            raise ValueError("piece_chunks must be >= 1")
        self.fmt = fmt
        self.side_key = {1: "cdf", 2: "rec", 3: "side3"}[fmt]
        self.L, self.T, self.C = L, T, C_
        self.bins_k = bins_k
        self.bins_v = bins_k if bins_v is None else bins_v
        self.levels = [(self.bins_k, self.bins_v)] if levels is None else \
            [(bk, bk if bv is None else bv) for bk, bv in levels]
        step = piece_chunks * chunk_tokens
        self.ranges = [(t0, min(T, t0 + step)) for t0 in range(0, T, step)]
        dev = torch.device(device)
        self.k = torch.empty((L, T, C_), dtype=torch.float16, device=dev)
        self.v = torch.empty((L, T, C_), dtype=torch.float16, device=dev)
        mk = lambda t0, t1, bk, bv: _codec.Codec(L, t1 - t0, C_, bk, bv, chunk_tokens=chunk_tokens, device=dev,
                                                 fmt=fmt, group=group)
        # [level][piece]
        self.enc = [[mk(t0, t1, bk, bv) for t0, t1 in self.ranges] for bk, bv in self.levels]
        self.dec = [[mk(t0, t1, bk, bv) for t0, t1 in self.ranges] for bk, bv in self.levels]
        self.host = []
        for lv_codecs in self.enc:
            hl = []
            for cd in lv_codecs:
                o = cd.out
                pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                side = getattr(o, self.side_key)
                hl.append({"packed": torch.empty(cd.capacity, dtype=torch.uint8, pin_memory=True),
                           "len": pin(o.len), "off": pin(o.off), self.side_key: pin(side), "max1": pin(o.max1)})
            self.host.append(hl)
        self.level = [0] * len(self.ranges)  # each piece's level in the current pass
        self.n_host = torch.zeros(len(self.ranges), dtype=torch.int64, pin_memory=True)
        # format 3: each piece's count bytes |V| (the uint64 after its slice offsets)
        self.v3_host = torch.zeros(len(self.ranges), dtype=torch.int64, pin_memory=True)
        self.status_host = torch.zeros(2 * len(self.ranges), dtype=torch.int32, pin_memory=True)
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_code = torch.cuda.Stream(device=dev)
        self.s_n = torch.cuda.Stream(device=dev)    # byte counts (kept off s_out: each waits on its piece)
        self.s_out = torch.cuda.Stream(device=dev)
        self.s_rx = torch.cuda.Stream(device=dev)
        self.s_dec = torch.cuda.Stream(device=dev)
        ev = lambda: [torch.cuda.Event() for _ in self.ranges]
        self.ev_in, self.ev_enc, self.ev_n, self.ev_out, self.ev_rx = ev(), ev(), ev(), ev(), ev()
        self.ev_done = torch.cuda.Event()

    # -- sender ---------------------------------------------------------------
    def _copy_in(self, dst: torch.Tensor, src: torch.Tensor, t0: int, t1: int):
        rt = _cudart()
        row = self.C * 2
        pitch = self.T * row
        err = rt.cudaMemcpy2DAsync(C.c_void_p(dst.data_ptr() + t0 * row), pitch,
                                   C.c_void_p(src.data_ptr() + t0 * row), pitch, (t1 - t0) * row, self.L,
                                   _MEMCPY_H2D, C.c_void_p(self.s_in.cuda_stream))
        if err != 0:
            raise RuntimeError(f"cudaMemcpy2DAsync failed ({err})")

    def _send(self, p: int, k_host: torch.Tensor, v_host: torch.Tensor, level: int = 0):
        t0, t1 = self.ranges[p]
        self.level[p] = level
        enc = self.enc[level][p]
        self._copy_in(self.k, k_host, t0, t1)
        self._copy_in(self.v, v_host, t0, t1)
        self.ev_in[p].record(self.s_in)
        self.s_code.wait_event(self.ev_in[p])
        enc.compress(self.k[:, t0:t1], self.v[:, t0:t1], stream=self.s_code)
        self.ev_enc[p].record(self.s_code)
        self.s_n.wait_event(self.ev_enc[p])
        _copy(self.n_host[p:p + 1], enc.out.off[-1:], 8, self.s_n)
        if self.fmt == 3:
            o = enc.out
            ns = 2 * self.L * (-(-(o.T) // o.chunk_tokens))
            _copy(self.v3_host[p:p + 1], o.side3[8 * ns:8 * ns + 8], 8, self.s_n)
        self.ev_n[p].record(self.s_n)

    def stream_pieces(self, k_host: torch.Tensor, v_host: torch.Tensor, ahead: int = 2, policy=None):
        """fp16 [L, T, C] pinned host K, V -> compressed pieces in pinned host
        memory, yielded in order as soon as each piece's copy-out is enqueued
        (its `ready` event marks the bytes on the host). Input copies run
        `ahead` pieces in front of the piece being yielded, so copies a
        consumer enqueues for piece p (the receiver's) take their place in the
        host-to-device queue behind piece p + ahead's input rather than behind
        every input. policy: None (level 0), or an object with
        level_for(tokens) -> level and observe(level, tokens, nbytes) (e.g.
        AdaptiveLevels), asked when a piece is sent and told its size."""
        if policy is None:
            choose = lambda p: 0
        else:
            choose = lambda p: int(policy.level_for(self.ranges[p][1] - self.ranges[p][0]))
        for t in (k_host, v_host):
            if t.device.type != "cpu" or not t.is_pinned() or t.dtype != torch.float16 or not t.is_contiguous():
                raise ValueError("K and V must be contiguous pinned host fp16 tensors")
            if tuple(t.shape) != (self.L, self.T, self.C):
                raise ValueError("K/V shape differs from the streamer's")
        npc = len(self.ranges)
        ahead = max(1, ahead)
        for p in range(min(ahead, npc)):
            self._send(p, k_host, v_host, self._checked(choose(p)))
        for p, (t0, t1) in enumerate(self.ranges):
            self.ev_n[p].synchronize()  # the piece's byte count, needed to size its copy
            n = int(self.n_host[p])
            lv = self.level[p]
            o, h = self.enc[lv][p].out, self.host[lv][p]
            self.s_out.wait_event(self.ev_enc[p])
            _copy(h["packed"], o.packed, n, self.s_out)
            side_bytes = 0
            if self.fmt == 3:  # the side buffer's used bytes; offsets stay behind (rebuilt from the lengths)
                side_bytes = o.side3_fixed + int(self.v3_host[p])
                keys = ("len", "max1")
                _copy(h["side3"], o.side3, side_bytes, self.s_out)
            else:
                keys = ("len", "off", self.side_key, "max1")
            for key in keys:
                _copy(h[key], getattr(o, key), _nb(h[key]), self.s_out)
            _copy(self.status_host[2 * p:2 * p + 1], o.status, 4, self.s_out)
            self.ev_out[p].record(self.s_out)
            if policy is not None:
                policy.observe(lv, t1 - t0, n + (side_bytes if self.fmt == 3 else _nb(h[self.side_key])))
            yield HostPiece(t0, t1, n, h["packed"], h["len"], h["off"], h[self.side_key], h["max1"], self.ev_out[p],
                            self.fmt, side_bytes, lv)
            if p + ahead < npc:
                self._send(p + ahead, k_host, v_host, self._checked(choose(p + ahead)))

    def _checked(self, level: int) -> int:
        if not 0 <= level < len(self.levels):
            raise ValueError(f"level {level} outside the {len(self.levels)} configured")
        return level

    def compress_from_host(self, k_host: torch.Tensor, v_host: torch.Tensor, policy=None) -> list[HostPiece]:
        """All pieces of `stream_pieces` (returns once every copy-out is enqueued)."""
        return list(self.stream_pieces(k_host, v_host, policy=policy))

    # -- receiver -------------------------------------------------------------
    def receive(self, p: int, hp: HostPiece, upload: torch.cuda.Stream | None = None):
        """Piece p (host) -> fp32 [L, t1 - t0, C] K, V on the device: copy in on
        `upload` (default: the receiver's own stream) once the piece is on the
        host, decompress on the decoding stream, status word back to the host."""
        cd = self.dec[hp.level][p]
        rx = cd.out
        up = self.s_rx if upload is None else upload
        up.wait_event(hp.ready)
        _copy(rx.packed, hp.packed, hp.nbytes, up)
        if self.fmt == 3:
            for key in ("len", "max1"):
                _copy(getattr(rx, key), getattr(hp, key), _nb(getattr(hp, key)), up)
            _copy(rx.side3, hp.side, hp.side_bytes, up)
        else:
            for key in ("len", "off", "max1"):
                _copy(getattr(rx, key), getattr(hp, key), _nb(getattr(hp, key)), up)
            _copy(getattr(rx, self.side_key), hp.side, _nb(hp.side), up)
        self.ev_rx[p].record(up)
        self.s_dec.wait_event(self.ev_rx[p])
        out = cd.decompress(rx, stream=self.s_dec)
        _copy(self.status_host[2 * p + 1:2 * p + 2], cd.dstatus, 4, self.s_dec)
        return out

    def decompress_from_host(self, pieces, upload: torch.cuda.Stream | None = None):
        """Every piece through `receive`; `pieces` may be the `stream_pieces`
        generator, so each piece's receive is enqueued as soon as it exists.
        Returns the list of (out_k, out_v) and the event that marks the last
        decompression (and the status words in `status_host`) done."""
        outs = [self.receive(p, hp, upload) for p, hp in enumerate(pieces)]
        self.ev_done.record(self.s_dec)
        return outs, self.ev_done

    def roundtrip(self, k_host: torch.Tensor, v_host: torch.Tensor, policy=None):
        """Compress from host, ship each piece to the host and back, decompress:
        returns (pieces, outs, done event), receiver work enqueued piece by piece
        as the sender produces them. The uploads share the input-copy stream, so
        the host-to-device queue alternates: input p + 2 waits behind upload p."""
        pieces = []

        def gen():
            for hp in self.stream_pieces(k_host, v_host, policy=policy):
                pieces.append(hp)
                yield hp
        outs, done = self.decompress_from_host(gen(), upload=self.s_in)
        return pieces, outs, done

    def status(self) -> int:
        """OR of every piece's compress and decompress status words (call
        after the returned event has completed)."""
        return int(np.bitwise_or.reduce(self.status_host.numpy()))

    def bytes_moved(self, pieces: list[HostPiece]) -> tuple[int, int]:
        """(host-to-device, device-to-host) bytes of one compress + decompress."""
        fp16 = 2 * 2 * self.L * self.T * self.C
        if self.fmt == 3:
            side = sum(hp.len.numel() * 4 + hp.side_bytes + hp.max1.numel() * 2 for hp in pieces)
        else:
            side = sum(hp.len.numel() * 4 + hp.off.numel() * 8 + _nb(hp.side) + hp.max1.numel() * 2
                       for hp in pieces)
        comp = sum(hp.nbytes for hp in pieces)
        return fp16 + comp + side, 8 * len(pieces) + comp + side + 8 * len(pieces)
