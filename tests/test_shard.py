"""Sharding by chunk ranges: the ranks' outputs, joined, are byte-identical to
one call over the whole tensor (chunks are coded independently, [CG §1.2(4)]).
The per-rank coding here is the oracle's; the GPU form of the same check is in
test_gpu_shard.py."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from kv_cache_compression_cg_gb300 import shard


def _input(L, T, C_, seed):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((L, T, C_)) * rng.lognormal(0, 0.5, (1, 1, C_))).astype(np.float16)
    v = (rng.standard_normal((L, T, C_)) * 0.5).astype(np.float16)
    return k, v


def _part(oracle_mod, k, v, Tc, bins_k, bins_v, t0, t1):
    if t1 == t0:  # a rank left without chunks contributes nothing
        L = k.shape[0]
        return {"max1": np.zeros((2, L, 0), np.uint16), "cdf": np.zeros(0, np.uint16),
                "packed": np.zeros(0, np.uint8), "len": np.zeros(0, np.uint32),
                "off": np.zeros(1, np.uint64)}
    out = oracle_mod.compress(np.ascontiguousarray(k[:, t0:t1]), np.ascontiguousarray(v[:, t0:t1]),
                              Tc, bins_k, bins_v)
    return {n: out[n] for n in ("max1", "cdf", "packed", "len", "off")}


def _same(a, b):
    return all(np.array_equal(a[n], b[n]) for n in ("max1", "cdf", "packed", "len", "off"))


@pytest.mark.parametrize("n_chunks,world", [(0, 2), (1, 2), (4, 2), (5, 3), (7, 4), (3, 5)])
def test_chunk_ranges_partition(n_chunks, world):
    ranges = [shard.chunk_range(n_chunks, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n_chunks
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)


def test_token_ranges_on_chunk_boundaries():
    T, Tc = 1000, 256
    rs = [shard.token_range(T, Tc, 3, r) for r in range(3)]
    assert rs == [(0, 512), (512, 768), (768, 1000)]
    with pytest.raises(ValueError):
        shard.chunk_range(4, 2, 2)


@pytest.mark.parametrize("T,Tc,world", [(200, 64, 2), (200, 64, 3), (130, 32, 5), (64, 64, 2)])
def test_join_equals_whole(oracle_mod, T, Tc, world):
    L, C_ = 3, 40
    bins_k, bins_v = [32, 16, 8], [16, 16, 32]
    k, v = _input(L, T, C_, seed=T + world)
    whole = _part(oracle_mod, k, v, Tc, bins_k, bins_v, 0, T)
    parts = [_part(oracle_mod, k, v, Tc, bins_k, bins_v, *shard.token_range(T, Tc, world, r))
             for r in range(world)]
    assert _same(shard.assemble(parts), whole)


def test_join_detects_a_wrong_order(oracle_mod):
    L, T, C_, Tc = 2, 128, 16, 32
    k, v = _input(L, T, C_, seed=7)
    whole = _part(oracle_mod, k, v, Tc, [32, 32], [32, 32], 0, T)
    parts = [_part(oracle_mod, k, v, Tc, [32, 32], [32, 32], *shard.token_range(T, Tc, 2, r))
             for r in range(2)]
    assert not _same(shard.assemble(parts[::-1]), whole)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_path):
    import torch.distributed as dist
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        L, T, C_, Tc = 2, 300, 48, 64
        bins_k, bins_v = [32, 16], [32, 8]
        k, v = _input(L, T, C_, seed=11)
        t0, t1 = shard.token_range(T, Tc, world, rank)
        mine = _part(oracle, k, v, Tc, bins_k, bins_v, t0, t1)
        base, grand, totals = shard.exchange_totals(int(mine["off"][-1]))
        parts = [None] * world
        dist.all_gather_object(parts, mine)
        if rank == 0:
            whole = _part(oracle, k, v, Tc, bins_k, bins_v, 0, T)
            joined = shard.assemble(parts)
            ok = (_same(joined, whole) and grand == int(whole["off"][-1])
                  and base == 0 and totals == [int(p["off"][-1]) for p in parts])
            with open(result_path, "w") as fh:
                fh.write("ok" if ok else "mismatch")
        else:
            # this rank's bytes start where the lower ranks' bytes end
            assert base == sum(totals[:rank])
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_join_equals_whole(oracle_mod, tmp_path):
    result = tmp_path / "result.txt"
    mp.spawn(_rank_main, args=(2, _free_port(), str(result)), nprocs=2, join=True)
    assert result.read_text() == "ok"
