"""Chunk-range sharding on the GPU: token-range views of one resident tensor,
each compressed by its own call (as the ranks of a multi-GPU job would), join
to exactly the bytes of one call over the whole tensor, and each range
decompresses to the whole call's output rows."""
import numpy as np
import pytest
import torch

from kv_cache_compression_cg_gb300 import shard

pytestmark = pytest.mark.gpu


def _host(out, cd):
    nstreams = cd.nstreams
    total = int(out.off[-1].item())
    return {"max1": out.max1.cpu().numpy().view(np.uint16),
            "cdf": out.cdf[:cd.cdf_elems].cpu().numpy().view(np.uint16),
            "packed": out.packed[:total].cpu().numpy(),
            "len": out.len[:nstreams].cpu().numpy().view(np.uint32),
            "off": out.off.cpu().numpy().view(np.uint64)}


@pytest.mark.parametrize("name,world", [("mistral_chunk", 2), ("tiny", 2), ("ctx4096", 3)])
def test_ranges_join_to_whole(synth_mod, name, world):
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required")
    from kv_cache_compression_cg_gb300 import build, codec
    build.build()
    w = synth_mod.WORKLOADS[name]
    T = w.T if name != "mistral_chunk" else 200   # ragged last chunk
    Tc = w.chunk_tokens if name != "mistral_chunk" else 64
    k, v = synth_mod.generate_device(w, T=T)
    whole_cd = codec.Codec(w.L, T, w.C, w.bins_k, w.bins_v, chunk_tokens=Tc)
    whole = _host(whole_cd.compress(k, v), whole_cd)
    wk, wv = whole_cd.decompress()
    parts = []
    for r in range(world):
        t0, t1 = shard.token_range(T, Tc, world, r)
        cd = codec.Codec(w.L, t1 - t0, w.C, w.bins_k, w.bins_v, chunk_tokens=Tc)
        out = cd.compress(k[:, t0:t1], v[:, t0:t1])
        assert int(out.status.item()) == 0
        parts.append(_host(out, cd))
        ok, ov = cd.decompress()
        torch.cuda.synchronize()
        assert int(cd.dstatus.item()) == 0
        assert torch.equal(ok.view(torch.int32), wk[:, t0:t1].view(torch.int32))
        assert torch.equal(ov.view(torch.int32), wv[:, t0:t1].view(torch.int32))
    joined = shard.assemble(parts)
    for n in ("max1", "cdf", "packed", "len", "off"):
        assert np.array_equal(joined[n], whole[n]), n
