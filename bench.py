#!/usr/bin/env python3
"""Benchmark of the CacheGen KV codec on GB300: one step = compress
(quantise -> CDF -> range-encode -> pack) plus decompress (decode fused with
dequantisation) of one synthetic KV workload, resident in HBM.

Prints one JSON line. Default workload: K and V fp16 [32, 4096, 1024] in 16
chunks of 256 tokens (Llama-3.1-8B / Mistral-7B KV shape), bins 32 for layers
0-9 and 16 for 10-31, AR(1) rho=0.9 values with 2% outlier channels, seed 2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one rank per GPU; each rank codes its own copy of
the workload (seed + rank) with no collective on the data path (weak
scaling); rank 0 prints the line with the max over ranks of the timed region.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV encode & decode GB/s (fp16 in) at 1 GB300, % of HBM roofline; compression ratio"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024
KERNELS_PER_STEP = 4  # compress_init, compress_tma, pack, decode_pipe (the ctx4096 shape takes the fused paths);
# format 3 adds its side-buffer packing (3), the offset scan (3) and the record unpacking (1)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ctx4096")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--format", type=int, choices=[1, 2, 3], default=2,
                    help="side information: 1 = CDF entries, 2 = symbol-count records, "
                         "3 = compact count records (offsets rebuilt from the lengths)")
    ap.add_argument("--piece-chunks", type=int, default=2,
                    help="chunks per piece of the streamed end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-call figures of the other seeded workloads")
    ap.add_argument("--tokens", type=int, default=0,
                    help="code only the first N tokens of the workload (same bytes; for profiling a smaller case)")
    ap.add_argument("--no-chunk-parallel", action="store_true",
                    help="skip the oracle's chunk-parallel timing on all host cores")
    ap.add_argument("--group", type=int, default=1,
                    help="token-locality delta group size (1: none, the page's LMCache code path)")
    ap.add_argument("--bins", type=int, default=0,
                    help="the same bins for every layer of K and V instead of the workload's (a wider "
                         "alphabet on the same values; reports no committed traffic)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.idx)], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        self.out.flush()
        with open(self.out.name) as fh:
            rows = [r.strip().split(", ") for r in fh if r.strip()]
        os.unlink(self.out.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except (IndexError, ValueError):
                continue
            for n, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def alg_ops_encode() -> int:
    """Integer/fp32 operations the specification needs per symbol to compress:
    quantise (convert, multiply, add, round, clamp: 5), count (1), coder step
    (r = range >> 16, split the CDF entry into lo and f, low += r*lo with the
    carry into the pending bits, range = r*f: 6), renormalise (shift count from
    clz: 2, shift low into the pending bits, low, range, bit count: 4), group
    max (1) -> 19."""
    return 19


def alg_ops_decode(P: int) -> int:
    """Per symbol to decompress: r (1), binary search over the P-entry row
    (multiply, compare, select per step: 3 log2 P), clamp (1), code -= r*lo (1),
    range = r*f (1), shift count (2), shift code, bit buffer, range, bit count
    (4), dequantise (lookup, multiply: 2) -> 12 + 3 log2 P."""
    return 12 + 3 * (P.bit_length() - 1)


def kernel_traffic(kernel: str, sources):
    """DRAM bytes per launch from the committed ncu table, only while the
    kernel's sources still hash to the values recorded with the counters."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", "traffic.md")
    csrc = os.path.join(ROOT, "kv_cache_compression_cg_gb300", "csrc")
    try:
        with open(path) as fh:
            text = fh.read()
        h = hashlib.sha256()
        for name in sources:
            with open(os.path.join(csrc, name), "rb") as fh:
                h.update(fh.read())
        digest = h.hexdigest()[:16]
    except OSError:
        return None
    for m in re.finditer(r"^\|\s*(\w+)\s*\|\s*([0-9]+)\s*\|\s*([0-9a-f]{16})\s*\|", text, re.M):
        if m.group(1) == kernel and m.group(3) == digest:
            return int(m.group(2))
    return None


def workload_config(w, extra=None):
    cfg = {"workload": w.name, "shape_per_kv": [w.L, w.T, w.C], "chunk_tokens": w.chunk_tokens,
           "bins_k": sorted(set(w.bins_k)), "bins_layer_split": sum(1 for b in w.bins_k if b == max(w.bins_k)),
           "values": w.describe(), "l2": "inputs > L2 and an L2-sized buffer written between timed steps"}
    if extra:
        cfg.update(extra)
    return cfg


def side_bytes(cd, out, w, fmt):
    """Side information that travels with the streams: CDF entries, count
    records or the format 3 side buffer; max1; lengths; offsets (format 3
    rebuilds them from the lengths)."""
    side_info = {1: 2 * cd.cdf_elems, 2: cd.rec_bytes}.get(fmt) or out.side3_bytes()
    return side_info + 2 * 2 * w.L * w.T + 4 * cd.nstreams + (8 * (cd.nstreams + 1) if fmt < 3 else 0)


WORKLOAD_SET = ("tiny", "mistral_chunk", "uniform", "ctx32k", "stress80k")


def other_workloads(args, hbm, flush, skip):
    """Per-call compress and decompress figures of the other seeded workloads
    (inputs from the device generator, resident in HBM; each call timed alone
    with CUDA events on the launching stream, an L2-sized buffer written
    before each; mean of 5 after 3 warm-ups)."""
    import torch
    from kv_cache_compression_cg_gb300 import codec, synth
    stream = torch.cuda.current_stream()
    res = {}
    for name in WORKLOAD_SET:
        if name == skip:
            continue
        w = synth.WORKLOADS[name]
        k, v = synth.generate_device(w)
        cd = codec.Codec(w.L, w.T, w.C, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens, fmt=args.format,
                         group=args.group)
        for _ in range(3):
            cd.compress(k, v)
            cd.decompress()
        torch.cuda.synchronize()

        def timed(fn):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
            for a, b in evs:
                flush.zero_()
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
            return statistics.mean(a.elapsed_time(b) for a, b in evs)

        cms = timed(lambda: cd.compress(k, v))
        dms = timed(cd.decompress)
        out = cd.out
        total = out.total_bytes()
        status = int(out.status.item()) | int(cd.dstatus.item())
        n_el = 2 * w.L * w.T * w.C
        fp16 = 2 * n_el
        side = side_bytes(cd, out, w, args.format)
        c_alg, d_alg = fp16 + total + side, total + side + 4 * n_el
        res[name] = {
            "shape_per_kv": [w.L, w.T, w.C], "chunks": w.n_chunks, "slices": 2 * w.L * w.n_chunks,
            "compress_ms": cms, "decompress_ms": dms,
            "compress_gbs": fp16 / (cms * 1e-3) / 1e9, "decompress_gbs": fp16 / (dms * 1e-3) / 1e9,
            "compress_frac_of_hbm": {"fp16_in": fp16 / (cms * 1e-3) / 1e9 / hbm,
                                     "algorithmic": c_alg / (cms * 1e-3) / 1e9 / hbm},
            "decompress_frac_of_hbm": {"fp16_in": fp16 / (dms * 1e-3) / 1e9 / hbm,
                                       "algorithmic": d_alg / (dms * 1e-3) / 1e9 / hbm},
            "compression_ratio": {"total": fp16 / (total + side), "payload": fp16 / total,
                                  "bits_per_symbol": 8 * total / n_el},
            "status_word": status,
        }
        del cd, k, v, out
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, single thread, on a bounded sample
# ---------------------------------------------------------------------------
def oracle_step_time(k, v, w, tokens, fmt=2, group=1):
    import oracle
    ks = k[:, :tokens].copy()
    vs = v[:, :tokens].copy()
    t0 = time.perf_counter()
    if fmt == 3:
        r = oracle.compress_v3(ks, vs, w.chunk_tokens, w.bins_k, w.bins_v, group=group)
        oracle.decompress_v3(r["packed"], r["len"], r["side"], r["max1"], w.L, tokens, w.C, w.chunk_tokens,
                             w.bins_k, w.bins_v, group=group)
    elif group > 1:
        r = oracle.compress_ex(ks, vs, w.chunk_tokens, w.bins_k, w.bins_v, fmt=fmt, group=group)
        oracle.decompress_ex(r["packed"], r["off"], r["len"], r["cdf" if fmt == 1 else "rec"], r["max1"], w.L,
                             tokens, w.C, w.chunk_tokens, w.bins_k, w.bins_v, fmt=fmt, group=group)
    elif fmt == 2:
        r = oracle.compress_v2(ks, vs, w.chunk_tokens, w.bins_k, w.bins_v)
        oracle.decompress_v2(r["packed"], r["off"], r["len"], r["rec"], r["max1"], w.L, tokens, w.C,
                             w.chunk_tokens, w.bins_k, w.bins_v)
    else:
        r = oracle.compress(ks, vs, w.chunk_tokens, w.bins_k, w.bins_v)
        oracle.decompress(r["packed"], r["off"], r["len"], r["cdf"], r["max1"], w.L, tokens, w.C,
                          w.chunk_tokens, w.bins_k, w.bins_v)
    dt = time.perf_counter() - t0
    return dt, ks.nbytes + vs.nbytes


def _chunk_worker(name, chunk, fmt, group, reps, barrier, results):
    """One process of the chunk-parallel timing: regenerates its own chunk of
    the workload, then times the oracle on it once per repetition, all
    processes released together by the barrier."""
    import numpy as np
    from kv_cache_compression_cg_gb300 import synth
    w = synth.WORKLOADS[name]
    t0 = chunk * w.chunk_tokens
    t1 = min(w.T, t0 + w.chunk_tokens)
    k = np.stack([synth.generate_slice_range(w, 0, l, t0, t1) for l in range(w.L)])
    v = np.stack([synth.generate_slice_range(w, 1, l, t0, t1) for l in range(w.L)])
    for _ in range(reps):
        barrier.wait()
        dt, nbytes = oracle_step_time(k, v, w, t1 - t0, fmt, group)
        results.put((chunk, dt, nbytes))


def oracle_chunk_parallel(w, fmt=2, group=1, reps=3, workers=None):
    """The oracle, unchanged, run by one process per host core over
    independent chunks (worker i codes chunk i mod the chunk count), each
    compress + decompress timed between a common start and the last finish.
    Processes are spawned (no fork of a process that has a CUDA context)."""
    import multiprocessing as mp
    if workers is None:
        workers = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(workers + 1)
    results = ctx.Queue()
    procs = [ctx.Process(target=_chunk_worker, args=(w.name, i % w.n_chunks, fmt, group, reps, barrier, results))
             for i in range(workers)]
    for p in procs:
        p.start()
    walls, nbytes = [], 0
    try:
        for _ in range(reps):
            barrier.wait(timeout=600)
            t0 = time.perf_counter()
            got = [results.get(timeout=600) for _ in range(workers)]
            walls.append(time.perf_counter() - t0)
            nbytes = sum(g[2] for g in got)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    wall = statistics.median(walls)
    return {"value": nbytes / wall / 1e9, "unit": UNIT, "cores": workers, "kind": "oracle, chunk-parallel",
            "sample": f"{workers} processes, one {w.chunk_tokens}-token chunk each (compress + decompress), "
                      f"median of {reps} repetitions"}


def run_reference(args):
    """--impl reference: the CPU oracle (the only reference implementation of
    this method here) timed on the host cores, on bounded samples."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from kv_cache_compression_cg_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.bins:
        w = dataclasses.replace(w, bins_k=(args.bins,) * w.L, bins_v=(args.bins,) * w.L)
    tokens = min(w.T, w.chunk_tokens)
    k, v = synth.generate(w, T=tokens)
    for _ in range(args.warmup):
        oracle_step_time(k, v, w, tokens, args.format, args.group)
    times = []
    nbytes = 0
    for _ in range(args.steps):
        dt, nbytes = oracle_step_time(k, v, w, tokens, args.format, args.group)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = nbytes / (ms * 1e-3) / 1e9
    sample = f"first chunk ({tokens} tokens x {w.L} layers x {w.C} channels, K and V) per step"
    cpu = {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample}
    if not args.no_chunk_parallel:
        cpu["chunk_parallel"] = oracle_chunk_parallel(w, args.format, args.group)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, {"sample": sample, "format": args.format, "delta_group": args.group}),
        "cpu_baseline": cpu,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from kv_cache_compression_cg_gb300 import build as cuda_build
    if rank == 0:
        cuda_build.build()
    if world > 1:
        dist.barrier()
    from kv_cache_compression_cg_gb300 import codec, synth

    base = synth.WORKLOADS[args.workload]
    if args.tokens:
        base = dataclasses.replace(base, T=min(args.tokens, base.T))
    if args.bins:
        base = dataclasses.replace(base, bins_k=(args.bins,) * base.L, bins_v=(args.bins,) * base.L)
    w = dataclasses.replace(base, seed=base.seed + 1000 * rank) if rank else base
    k, v = synth.generate_device(w)  # same bytes as the host generator
    fp16_bytes = 2 * k.numel() * k.element_size()
    k_pin = torch.empty(k.shape, dtype=k.dtype, pin_memory=True)
    v_pin = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
    k_pin.copy_(k)
    v_pin.copy_(v)
    k_h, v_h = k_pin.numpy(), v_pin.numpy()
    stream = torch.cuda.current_stream()
    cd = codec.Codec(w.L, w.T, w.C, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens, fmt=args.format,
                     group=args.group)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")

    def step():
        cd.compress(k, v)
        cd.decompress()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    out = cd.out
    total = out.total_bytes()
    status = int(out.status.item()) | int(cd.dstatus.item())
    # reconstruction error of the output (reported, outside any timed region)
    rk, rv = cd.decompress()
    rel_rmse = {name: float((((o - x.float()) ** 2).mean() / (x.float() ** 2).mean()).sqrt())
                for name, o, x in (("k", rk, k), ("v", rv, v))}

    # timed region
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        cd.compress(k, v)
        ev[i][1].record(stream)
        cd.decompress()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    comp_ms = [a.elapsed_time(b) for a, b, _ in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    step_ms = sum(comp_ms) / len(comp_ms) + sum(dec_ms) / len(dec_ms)
    region_ms = sum(comp_ms) + sum(dec_ms)
    if world > 1:
        t = torch.tensor([region_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        region_ms = float(t.item())
        dist.barrier()
    hbm, peak_kind = peaks()

    # Per-call device time on the launching stream. cg_decompress_chunk is one
    # kernel (k_decode_pipe); cg_compress_chunk is k_compress_init (zeroing the
    # look-back slots, a few microseconds) followed by k_compress_tma.
    def time_call(fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    comp_kernel_ms = time_call(lambda: cd.compress(k, v))
    dec_kernel_ms = time_call(cd.decompress)
    n_el = 2 * w.L * w.T * w.C
    side = side_bytes(cd, out, w, args.format)
    dec_alg_bytes = total + side + 4 * n_el
    comp_alg_bytes = fp16_bytes + total + side
    A = max(max(w.bins_k), max(w.bins_v))
    if args.format >= 2:  # the largest layer alphabet, 2 * MAX + 1
        A = max(2 * (b // 2 - 1) + 1 for b in list(w.bins_k) + list(w.bins_v))
    P = 1 << (A - 1).bit_length()
    props = torch.cuda.get_device_properties(local)
    max_mhz = clocks.get("sm_max_mhz") or 2070.0
    # issue peak: SMs x 4 schedulers x one 32-lane instruction per cycle
    peak_tops = props.multi_processor_count * 4 * 32 * max_mhz * 1e6 / 1e12
    kern = {
        "compress": ("k_compress_tma (quantise + CDF + encode + pack)", comp_kernel_ms,
                     alg_ops_encode(), comp_alg_bytes, ["compress.cu", "coder.cuh", "cg_internal.cuh"]),
        "decompress": ("k_decode_pipe (decode + dequantise)", dec_kernel_ms,
                       alg_ops_decode(P), dec_alg_bytes, ["decode_pipe.cuh", "decode.cu", "cg_internal.cuh"]),
    }
    def roof(which):
        kname, kms, ops, kbytes, srcs = kern[which]
        achieved = kbytes / (kms * 1e-3) / 1e9
        alu = n_el * ops / (kms * 1e-3) / 1e12
        return {
            "kernel": kname, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind ==
            "measured" else "fallback", "algorithmic_bytes": kbytes, "ms": kms,
            "traffic": None if args.bins else kernel_traffic(
                f"{kname.split()[0]}_{args.workload}_f{args.format}_g{args.group}", srcs),
            "alu": {"achieved": alu, "peak": peak_tops, "unit": "Tops/s", "frac": alu / peak_tops,
                    "ops_per_symbol": ops,
                    "peak_kind": f"derived: {props.multi_processor_count} SMs x 4 schedulers x 32 lanes x "
                                 f"{max_mhz:g} MHz"},
        }

    dom = "compress" if comp_kernel_ms >= dec_kernel_ms else "decompress"
    roofline = roof(dom)
    rooflines = {"compress": roof("compress"), "decompress": roof("decompress")}

    comp_gbs = fp16_bytes / (statistics.mean(comp_ms) * 1e-3) / 1e9
    dec_gbs = fp16_bytes / (statistics.mean(dec_ms) * 1e-3) / 1e9
    value = world * fp16_bytes / (region_ms / args.steps * 1e-3) / 1e9

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": region_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "dtype_detail": "fp16 K/V in; binary32 quantise and dequantise; 32-bit integer range coder; "
                        "binary32 K/V out",
        "data": "synthetic",
        "config": workload_config(w, {"parallelism": f"chunk-sharded x{world}" if world > 1 else "1 GPU",
                                      "format": args.format, "delta_group": args.group}),
        "compress_gbs": comp_gbs, "decompress_gbs": dec_gbs,
        "compress_ms": statistics.mean(comp_ms), "decompress_ms": statistics.mean(dec_ms),
        "compress_frac_of_hbm": {"fp16_in": comp_gbs / hbm,
                                 "algorithmic": comp_alg_bytes / (statistics.mean(comp_ms) * 1e-3) / 1e9 / hbm},
        "decompress_frac_of_hbm": {"fp16_in": dec_gbs / hbm,
                                   "algorithmic": dec_alg_bytes / (statistics.mean(dec_ms) * 1e-3) / 1e9 / hbm},
        "compression_ratio": {"total": fp16_bytes / (total + side), "payload": fp16_bytes / total,
                              "bits_per_symbol": 8 * total / n_el},
        "roofline": roofline, "rooflines": rooflines,
        "reconstruction_rel_rmse": rel_rmse,
        "status_word": status, "clocks": clocks, "wall_s_timed_region": wall,
        "gpu_launches": (KERNELS_PER_STEP + (7 if args.format == 3 else 0)) * args.steps,
    }

    if not args.no_e2e:
        result["e2e"] = e2e(args, w, cd, k_pin, v_pin, fp16_bytes)
    if rank == 0 and world == 1 and not args.no_workloads:
        result["workloads"] = other_workloads(args, hbm, flush, args.workload)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_dt, cpu_bytes = oracle_step_time(k_h, v_h, w, min(w.T, 2 * w.chunk_tokens), args.format, args.group)
        reps = max(1, int(10.0 / max(cpu_dt, 1e-3)))
        times = [cpu_dt]
        for _ in range(min(reps, 20) - 1):
            times.append(oracle_step_time(k_h, v_h, w, min(w.T, 2 * w.chunk_tokens), args.format, args.group)[0])
        cpu_gbs = cpu_bytes / statistics.mean(times) / 1e9
        result["cpu_baseline"] = {
            "value": cpu_gbs, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {min(w.T, 2 * w.chunk_tokens)} tokens (compress + decompress), "
                      f"{len(times)} repetitions"}
        if not args.no_chunk_parallel:
            result["cpu_baseline"]["chunk_parallel"] = oracle_chunk_parallel(w, args.format, args.group)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def e2e(args, w, cd, k_pin, v_pin, fp16_bytes):
    """Through the public streaming API with host buffers: pinned fp16 K, V go
    in piece by piece (runs of whole chunks) while earlier pieces compress;
    each compressed piece comes back to pinned host memory as it is done; the
    receiver copies each piece back in and decompresses it, and the status
    words come back to the host. One step = all of that for the whole tensor;
    the decompressed output is checked once against the single-call result."""
    import torch
    from kv_cache_compression_cg_gb300.stream import StreamingCodec
    sc = StreamingCodec(w.L, w.T, w.C, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens, fmt=args.format,
                        piece_chunks=args.piece_chunks, group=args.group)
    times = []
    pieces = outs = None
    for i in range(max(args.warmup, 3) + args.steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pieces, outs, done = sc.roundtrip(k_pin, v_pin)
        done.synchronize()
        if i >= max(args.warmup, 3):
            times.append(time.perf_counter() - t0)
    status = sc.status()
    # the streamed output equals the single-call one, piece by piece
    ref_k, ref_v = cd.decompress()
    torch.cuda.synchronize()
    exact = all(torch.equal(ok.view(torch.int32), ref_k[:, hp.t0:hp.t1].view(torch.int32)) and
                torch.equal(ov.view(torch.int32), ref_v[:, hp.t0:hp.t1].view(torch.int32))
                for (ok, ov), hp in zip(outs, pieces))
    h2d, d2h = sc.bytes_moved(pieces)
    # the median step: the host link is shared with other jobs on the machine, and a step that
    # overlaps their transfers runs several times slower (mean and max reported alongside)
    sec = statistics.median(times)
    return {"value": fp16_bytes / sec / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": sec * 1e3, "statistic": f"median of {len(times)} steps",
            "ms_per_step_mean": statistics.mean(times) * 1e3, "ms_per_step_max": max(times) * 1e3,
            "pieces": len(pieces),
            "status_word": status, "matches_single_call": exact,
            "path": "pinned host fp16 K,V -> per piece of %d chunks: copy in, compress, compressed piece "
                    "to pinned host -> copy back in, decompress -> status words to host (5 CUDA streams)"
                    % args.piece_chunks}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
