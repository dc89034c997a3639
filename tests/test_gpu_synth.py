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
