"""The codec's calls are asynchronous on the caller's stream with no host
synchronisation and no allocation inside, so a compress + decompress step can
be captured once in a CUDA graph and replayed. Replays must write exactly what
eager calls write, for the inputs in the captured buffers at replay time, in
all three side-information formats and with the token-locality delta."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cg():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from kv_cache_compression_cg_gb300 import build, codec
    build.build()
    return codec


def _snapshot(cd, out, ok, ov):
    n = out.total_bytes()
    side = {1: out.cdf, 2: out.rec}[cd.fmt] if cd.fmt < 3 else out.side3[:out.side3_bytes()]
    return [out.max1.clone(), side.clone(), out.len.clone(), out.off.clone(), out.packed[:n].clone(),
            ok.clone(), ov.clone(), out.status.clone(), cd.dstatus.clone()]


# T = 1024 (four chunks, 256 slices) takes the throughput kernels; T = 256 (one
# chunk, 64 slices) the latency-mode ones, whose packing is a programmatic
# dependent launch
@pytest.mark.parametrize("fmt,group,T", [(1, 1, 1024), (2, 1, 1024), (3, 1, 1024), (2, 10, 1024), (1, 1, 256),
                                         (2, 1, 256)])
def test_graph_replay_equals_eager(cg, synth_mod, fmt, group, T):
    w = synth_mod.WORKLOADS["ctx4096"]
    k0, v0 = synth_mod.generate_device(w, T=T)
    k1, v1 = synth_mod.generate_device(synth_mod.WORKLOADS["mistral_chunk"], T=T)  # other values, same shape
    cd = cg.Codec(w.L, T, w.C, w.bins_k, w.bins_v, chunk_tokens=w.chunk_tokens, fmt=fmt, group=group)
    k = k0.clone()
    v = v0.clone()

    # eager results for both inputs
    want = []
    for kk, vv in ((k0, v0), (k1, v1)):
        k.copy_(kk)
        v.copy_(vv)
        out = cd.compress(k, v)
        ok, ov = cd.decompress()
        torch.cuda.synchronize()
        assert int(out.status.item()) == 0 and int(cd.dstatus.item()) == 0
        want.append(_snapshot(cd, out, ok, ov))

    # capture one step (torch's capture stream is the current stream inside)
    k.copy_(k0)
    v.copy_(v0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on a side stream, as torch asks before a capture
        cd.compress(k, v)
        cd.decompress()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = cd.compress(k, v)
        ok, ov = cd.decompress()
    torch.cuda.synchronize()

    for idx, (kk, vv) in enumerate(((k0, v0), (k1, v1), (k0, v0))):
        k.copy_(kk)
        v.copy_(vv)
        for t in (out.packed, out.len, out.off, ok, ov):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        got = _snapshot(cd, out, ok, ov)
        for a, b in zip(got, want[idx % 2]):
            assert torch.equal(a, b), idx
