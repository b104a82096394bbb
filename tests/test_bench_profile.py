"""The benchmark's roofline `traffic`: DRAM bytes per launch from a committed ncu summary,
reported only while the summary was taken on the kernel source that runs (its recorded
hash matches), else null."""
import hashlib

import bench


def _hash():
    h = hashlib.sha256()
    for f in bench.TC_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()


def test_committed_profiles_are_well_formed():
    # both summaries the bench reads carry the two machine-readable fields; when taken on
    # the current kernel source, the default workload's traffic is at least its compulsory
    # bytes (A, B and C of bf16 8192^3)
    import re
    for workload, path in bench.PROFILES.items():
        text = open(path).read()
        assert re.search(r"dram_bytes_per_launch:\s*[0-9]+", text), workload
        assert re.search(r"kernel_source_sha256:\s*[0-9a-f]{64}", text), workload
    v = bench.profile_traffic("bf16_8192")
    assert v is None or v >= 3 * 8192 * 8192 * 2
    # workloads without a summary report null
    assert bench.profile_traffic("tf32_4096") is None


def test_stale_or_missing_summary_reports_null(tmp_path, monkeypatch):
    good = tmp_path / "good.md"
    good.write_text("dram_bytes_per_launch: 12345\nkernel_source_sha256: %s\n" % _hash())
    stale = tmp_path / "stale.md"
    stale.write_text("dram_bytes_per_launch: 12345\nkernel_source_sha256: %s\n" % ("0" * 64))
    partial = tmp_path / "partial.md"
    partial.write_text("dram_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "PROFILES", {"a": str(good), "b": str(stale), "c": str(partial),
                                            "d": str(tmp_path / "missing.md")})
    assert bench.profile_traffic("a") == 12345.0
    assert bench.profile_traffic("b") is None
    assert bench.profile_traffic("c") is None
    assert bench.profile_traffic("d") is None
