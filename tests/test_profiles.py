"""The committed profile summaries stay tied to the sources they describe: the
up-projection's DRAM traffic that bench.py reports is recorded against a
digest of the GEMM source, and bench.py reports no traffic once that source
has changed since the capture."""
import hashlib
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_record_matches_gemm_source():
    src = os.path.join(ROOT, "activation_sparse_transformer_gb300", "csrc", "gemm_tcgen05.cu")
    with open(src, "rb") as fh:
        digest = hashlib.sha256(fh.read()).hexdigest()[:16]
    rows = []
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.txt")) as fh:
        for line in fh:
            parts = line.split()
            if parts and not parts[0].startswith("#"):
                rows.append(parts)
    up = [r for r in rows if r[0] == "up_pack" and r[1] == "1b"]
    assert len(up) == 1
    assert os.path.exists(os.path.join(ROOT, "profiles", up[0][4]))
    import bench
    traffic, note = bench.ncu_traffic("up_pack", "1b")
    if up[0][2] == digest:
        assert traffic == float(up[0][3])
    else:   # the kernel changed since the counters were taken: bench reports none
        assert traffic is None and note.startswith("stale")


def test_profiles_are_text_only():
    for name in os.listdir(os.path.join(ROOT, "profiles")):
        assert os.path.splitext(name)[1] in (".md", ".txt"), name
