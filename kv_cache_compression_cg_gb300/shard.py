"""Sharding the codec over ranks by contiguous chunk ranges.

Chunks are coded independently: each has its own CDFs and its own per-token
streams ([CG §1.2(4)], chunk-wise processing; [CG §2.3(2)], CDFs per chunk).
The stream index is chunk-major, so the streams, lengths and CDF rows of a
contiguous chunk range form one contiguous slice of the whole tensor's output.
A rank therefore compresses its token range with no exchange at all; the one
step that needs every rank is placing the ranks' packed bytes in a single
global buffer, which needs the exclusive scan of the per-rank byte totals
(one 8-byte value per rank).

Everything here is host logic; the coding itself runs in the CUDA library on
each rank's own GPU.
"""
from __future__ import annotations

import numpy as np

__all__ = ["chunk_range", "token_range", "exchange_totals", "assemble"]


def chunk_range(n_chunks: int, world: int, rank: int) -> tuple[int, int]:
    """Chunks [k0, k1) of `rank`: contiguous, sizes differing by at most one,
    the larger ranges first."""
    if world < 1 or not 0 <= rank < world or n_chunks < 0:
        raise ValueError("need world >= 1, 0 <= rank < world, n_chunks >= 0")
    base, extra = divmod(n_chunks, world)
    k0 = rank * base + min(rank, extra)
    return k0, k0 + base + (1 if rank < extra else 0)


def token_range(T: int, chunk_tokens: int, world: int, rank: int) -> tuple[int, int]:
    """Tokens [t0, t1) of `rank`; every boundary but T is a chunk boundary, so
    the rank's chunks are exactly the whole tensor's chunks k0..k1-1."""
    if chunk_tokens < 1:
        raise ValueError("chunk_tokens must be >= 1")
    nch = -(-T // chunk_tokens)
    k0, k1 = chunk_range(nch, world, rank)
    return min(T, k0 * chunk_tokens), min(T, k1 * chunk_tokens)


def exchange_totals(local_total: int, group=None, device=None) -> tuple[int, int, list[int]]:
    """All-gather the ranks' packed byte totals; returns (this rank's byte
    offset in the global buffer, the global total, every rank's total)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    mine = torch.tensor([int(local_total)], dtype=torch.int64, device=device)
    every = [torch.zeros_like(mine) for _ in range(world)]
    dist.all_gather(every, mine, group=group)
    totals = [int(t.item()) for t in every]
    return sum(totals[:rank]), sum(totals), totals


def assemble(parts: list[dict]) -> dict:
    """Join per-rank outputs (in rank order) into the whole tensor's output.

    Each part holds host arrays of one rank's compress call on its token range:
    max1 uint16 [2][L][T_r], cdf uint16 (chunk-major; format 2: rec uint8
    count records, chunk-major too), packed uint8 (exactly
    off[-1] bytes), len uint32 [2 L T_r], off uint64 [2 L T_r + 1]. The result
    is byte-identical to compressing the whole tensor in one call.
    """
    if not parts:
        raise ValueError("no parts")
    base = 0
    offs = []
    for p in parts:
        off = np.asarray(p["off"], dtype=np.uint64)
        if int(off[-1]) != len(p["packed"]):
            raise ValueError("a part's packed bytes differ from its off[-1]")
        offs.append(off[:-1] + np.uint64(base))
        base += int(off[-1])
    offs.append(np.array([base], dtype=np.uint64))
    side = "cdf" if "cdf" in parts[0] else "rec"  # format 1 CDF entries or format 2 count records
    return {
        "max1": np.concatenate([np.asarray(p["max1"], np.uint16) for p in parts], axis=2),
        side: np.concatenate([np.asarray(p[side], np.uint16 if side == "cdf" else np.uint8) for p in parts]),
        "packed": np.concatenate([np.asarray(p["packed"], np.uint8) for p in parts]),
        "len": np.concatenate([np.asarray(p["len"], np.uint32) for p in parts]),
        "off": np.concatenate(offs),
    }
