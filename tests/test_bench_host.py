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
