"""The device generator writes exactly the host generator's bytes (the input
to the CUDA path and to the oracle must be the same tensors)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "mistral_chunk", "uniform", "stress80k"])
def test_device_generator_matches_host(synth_mod, name):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    w = synth_mod.WORKLOADS[name]
    T = min(w.T, 512)
    k_d, v_d = synth_mod.generate_device(w, T=T)
    k_h, v_h = synth_mod.generate(w, T=T)
    assert np.array_equal(k_d.cpu().numpy().view(np.uint16), k_h.view(np.uint16))
    assert np.array_equal(v_d.cpu().numpy().view(np.uint16), v_h.view(np.uint16))


@pytest.mark.parametrize("name", ["ctx4096", "ctx32k"])
def test_device_generator_full_size_matches_recorded_sha256(synth_mod, name):
    """The device generator's full-size inputs (the bench's) have the recorded
    SHA-256 (written from the host generator by tests/golden/make_synth_sha256.py)."""
    import hashlib
    from conftest import read_golden
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    want = {n: d for n, d in read_golden("synth_sha256.txt")}[name]
    k_d, v_d = synth_mod.generate_device(synth_mod.WORKLOADS[name])
    h = hashlib.sha256()
    h.update(k_d.cpu().numpy().tobytes())
    h.update(v_d.cpu().numpy().tobytes())
    assert h.hexdigest() == want
