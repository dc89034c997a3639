"""Write synth_sha256.txt: the SHA-256 of each seeded workload's K and V bytes
as the host generator produces them (fp16, [L][T][C], K then V). The hashes
pin the generator itself (the same bytes on every machine and in every run);
they are not expected values of the codec. Run from the repository root:
    python tests/golden/make_synth_sha256.py"""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from kv_cache_compression_cg_gb300 import synth  # noqa: E402


def digest(name: str) -> str:
    k, v = synth.generate(synth.WORKLOADS[name])
    h = hashlib.sha256()
    h.update(k.tobytes())
    h.update(v.tobytes())
    return h.hexdigest()


def main():
    synth.build()
    lines = ["# SHA-256 of each seeded workload's fp16 K then V bytes, host generator",
             "# (written by tests/golden/make_synth_sha256.py)",
             "# workload | sha256"]
    for name in ("tiny", "mistral_chunk", "ctx4096", "ctx32k", "stress80k", "uniform"):
        lines.append(f"{name} | {digest(name)}")
    with open(os.path.join(HERE, "synth_sha256.txt"), "w") as fh:
        fh.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
