"""Checks of the seeded input generator (not part of the codec)."""
import math

import numpy as np
import pytest


def test_elementary_functions(synth_mod):
    L = synth_mod.lib()
    rng = np.random.default_rng(0)
    for x in np.concatenate([rng.uniform(1e-300, 1, 200), rng.uniform(1, 1e6, 200), [1.0, 2.0, 0.5]]):
        assert abs(L.syn_ln(x) - math.log(x)) <= 8 * math.ulp(abs(math.log(x))) + 1e-15
    for x in rng.uniform(-20, 20, 400):
        assert abs(L.syn_expo(x) - math.exp(x)) <= 4 * math.ulp(math.exp(x))
    import ctypes as C
    c, s = C.c_double(), C.c_double()
    for u in np.concatenate([rng.uniform(0, 1, 400), [0.0, 0.25, 0.5, 0.75]]):
        L.syn_cis2pi(u, C.byref(c), C.byref(s))
        assert abs(c.value - math.cos(2 * math.pi * u)) < 1e-15
        assert abs(s.value - math.sin(2 * math.pi * u)) < 1e-15


def test_half_conversion_matches_numpy(synth_mod):
    L = synth_mod.lib()
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-8, 5, 2000),
                         [0.0, -0.0, 65504.0, 65519.99, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26]])
    for x in xs:
        assert L.syn_half(float(x)) == np.float16(x).view(np.uint16), x
    assert L.syn_half(1e6) == 0x7BFF and L.syn_half(-1e6) == 0xFBFF


def test_deterministic_and_thread_independent(synth_mod):
    w = synth_mod.WORKLOADS["tiny"]
    a = synth_mod.generate(w, nthreads=1)
    b = synth_mod.generate(w, nthreads=3)
    assert all((x.view(np.uint16) == y.view(np.uint16)).all() for x, y in zip(a, b))
    s = synth_mod.generate_slice(w, 1, 1)
    assert (s.view(np.uint16) == a[1][1].view(np.uint16)).all()


def test_token_prefix_is_stable(synth_mod):
    for name in ("mistral_chunk", "stress80k", "uniform"):
        w = synth_mod.WORKLOADS[name]
        full = synth_mod.generate_slice(w, 0, 3, T=96)
        pre = synth_mod.generate_slice(w, 0, 3, T=40)
        assert (full[:40].view(np.uint16) == pre.view(np.uint16)).all()


def test_statistics(synth_mod):
    w = synth_mod.WORKLOADS["mistral_chunk"]
    x = synth_mod.generate_slice(w, 0, 0).astype(np.float64)  # [256, 1024]
    # AR(1): lag-1 autocorrelation per channel near rho = 0.9
    a, b = x[:-1] - x[:-1].mean(0), x[1:] - x[1:].mean(0)
    rho = (a * b).sum(0) / np.sqrt((a * a).sum(0) * (b * b).sum(0))
    assert abs(np.median(rho) - 0.9) < 0.05
    # 2% of 1024 channels are outliers at x8: the top-20 channel scales stand out
    sd = x.std(0)
    top = np.sort(sd)[-20:]
    assert np.median(top) > 4 * np.median(sd)
    u = synth_mod.generate_slice(synth_mod.WORKLOADS["uniform"], 1, 0).astype(np.float64)
    assert u.min() >= 0 and u.max() <= 1 and abs(u.mean() - 0.5) < 0.01  # fp16 rounding can reach 1.0
    t = synth_mod.generate_slice(synth_mod.WORKLOADS["stress80k"], 0, 0, T=512).astype(np.float64)
    z = t / np.median(np.abs(t), axis=0)
    assert abs(np.corrcoef(z[:-1].ravel(), z[1:].ravel())[0, 1]) < 0.02


def _recorded_sha256():
    from conftest import read_golden
    return {name: digest for name, digest in read_golden("synth_sha256.txt")}


@pytest.mark.parametrize("name", ["tiny", "mistral_chunk", "uniform", "ctx4096"])
def test_generator_bytes_match_recorded_sha256(synth_mod, name):
    """The generator's output is pinned: the same bytes as recorded (written by
    tests/golden/make_synth_sha256.py), on this machine and any other."""
    import hashlib
    k, v = synth_mod.generate(synth_mod.WORKLOADS[name])
    h = hashlib.sha256()
    h.update(k.tobytes())
    h.update(v.tobytes())
    assert h.hexdigest() == _recorded_sha256()[name]
