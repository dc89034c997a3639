"""Host-side pieces of bench.py that need no GPU: the oracle's timings on the
host cores (single process and chunk-parallel)."""
import bench


def test_oracle_step_time_counts_input_bytes(synth_mod):
    w = synth_mod.WORKLOADS["tiny"]
    k, v = synth_mod.generate(w)
    for fmt in (1, 2, 3):
        dt, nbytes = bench.oracle_step_time(k, v, w, w.T, fmt)
        assert dt > 0 and nbytes == k.nbytes + v.nbytes


def test_chunk_parallel_runs_every_worker(synth_mod):
    w = synth_mod.WORKLOADS["tiny"]
    r = bench.oracle_chunk_parallel(w, fmt=2, group=1, reps=2, workers=2)
    assert r["cores"] == 2 and r["unit"] == bench.UNIT and r["value"] > 0
    assert "2 processes" in r["sample"]


def _run_bench(*args, env=None):
    import json
    import os
    import subprocess
    import sys
    e = dict(os.environ)
    e.update(env or {})
    p = subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py"), *args],
                       capture_output=True, text=True, timeout=600, env=e)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_prints_one_contract_line():
    (d,) = _run_bench("--impl", "reference", "--steps", "2", "--warmup", "3", "--workload", "tiny",
                      "--format", "3")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny" and d["config"]["format"] == 3
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["value"] == d["value"] and cb["kind"] == "oracle" and cb["cores"] == 1
    assert cb["chunk_parallel"]["cores"] >= 1 and cb["chunk_parallel"]["value"] > 0


def test_reference_arm_silent_on_other_ranks():
    assert _run_bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--workload", "tiny",
                      "--no-chunk-parallel", env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


def test_bins_override_reaches_the_config():
    (d,) = _run_bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--workload", "tiny",
                      "--bins", "64", "--no-chunk-parallel")
    assert d["config"]["bins_k"] == [64]
