"""The committed profile summaries stay tied to the sources they describe: each
kernel's DRAM traffic that bench.py reports is recorded against a digest of
its source file, and bench.py reports no traffic once that source has changed
since the capture."""
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _records():
    rows = []
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.txt")) as fh:
        for line in fh:
            parts = line.split()
            if parts and not parts[0].startswith("#"):
                rows.append(parts)
    return rows


def test_traffic_records_follow_their_sources():
    import bench
    rows = _records()
    assert rows
    for kernel, workload, src, digest, nbytes, summary in (r[:6] for r in rows):
        assert os.path.exists(os.path.join(ROOT, "profiles", summary)), summary
        assert float(nbytes) > 0
        traffic, note = bench.ncu_traffic(kernel, workload)
        if bench.source_digest(src) == digest:
            assert traffic == float(nbytes)
        else:   # the kernel changed since the counters were taken: bench reports none
            assert traffic is None and note.startswith("stale")


def test_profiles_are_text_only():
    for name in os.listdir(os.path.join(ROOT, "profiles")):
        assert os.path.splitext(name)[1] in (".md", ".txt"), name


def test_digest_follows_code_not_comments():
    """A comment or blank-line edit keeps a capture's digest; any code edit
    (a literal with // in it included) changes it."""
    import bench
    base = 'int a = 1;  // x\nasm("mov // y");\n'
    same = '// header\nint a = 1;  // changed comment\n\nasm("mov // y");   \n'
    assert list(bench._code_lines(base)) == list(bench._code_lines(same))
    assert list(bench._code_lines(base)) != list(bench._code_lines('int a = 2;  // x\nasm("mov // y");\n'))
    assert list(bench._code_lines(base)) != list(bench._code_lines('int a = 1;  // x\nasm("mov // z");\n'))
