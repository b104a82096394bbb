"""The benchmark's roofline `traffic`: DRAM bytes per launch from a committed ncu summary,
reported only while the summary was taken on the kernel source that runs (its recorded
hash matches), else null."""
import hashlib

import bench


def _hash(sources=None):
    h = hashlib.sha256()
    for f in bench.TC_SOURCES if sources is None else sources:
        h.update(open(f, "rb").read())
    return h.hexdigest()


def test_committed_profiles_are_well_formed():
    # both summaries the bench reads carry the two machine-readable fields; when taken on
    # the current kernel source, the default workload's traffic is at least its compulsory
    # bytes (A, B and C of bf16 8192^3)
    import os
    import re
    for workload, (path, sources) in bench.PROFILES.items():
        if not os.path.exists(path):
            assert bench.profile_traffic(workload) is None
            continue
        text = open(path).read()
        has = (re.search(r"dram_bytes_per_launch:\s*[0-9]+", text),
               re.search(r"kernel_source_sha256:\s*[0-9a-f]{64}", text))
        if workload in ("bf16_8192", "bf16_skinny"):
            assert all(has), workload
        elif not all(has):  # a summary without the fields gives no traffic
            assert bench.profile_traffic(workload) is None
    v = bench.profile_traffic("bf16_8192")
    assert v is None or v >= 3 * 8192 * 8192 * 2
    # workloads without a summary report null
    assert bench.profile_traffic("f16acc_4096") is None


def test_stale_or_missing_summary_reports_null(tmp_path, monkeypatch):
    good = tmp_path / "good.md"
    good.write_text("dram_bytes_per_launch: 12345\nkernel_source_sha256: %s\n" % _hash())
    stale = tmp_path / "stale.md"
    stale.write_text("dram_bytes_per_launch: 12345\nkernel_source_sha256: %s\n" % ("0" * 64))
    partial = tmp_path / "partial.md"
    partial.write_text("dram_bytes_per_launch: 12345\n")
    src = bench.TC_SOURCES
    monkeypatch.setattr(bench, "PROFILES", {"a": (str(good), src), "b": (str(stale), src),
                                            "c": (str(partial), src),
                                            "d": (str(tmp_path / "missing.md"), src),
                                            "e": (str(good), bench.CHUNK_SOURCES)})
    assert bench.profile_traffic("a") == 12345.0
    assert bench.profile_traffic("b") is None
    assert bench.profile_traffic("c") is None
    assert bench.profile_traffic("d") is None
    assert bench.profile_traffic("e") is None  # taken on another kernel's sources


def test_clock_summary_bins_and_loaded_filter():
    line = "0, %d, 2070, %.1f, 0x0, Not Active, Not Active, Not Active, %s"
    text = "\n".join([line % (2070, 150.0, "Not Active")] +
                     [line % (mhz, 1390.0, "Active") for mhz in (1440, 1455, 1470, 1510)])
    s = bench.clock_summary(bench.parse_clock_samples(text), period_ms=50)
    assert s["samples"] == 5 and s["samples_under_load"] == 4
    assert s["sm_mhz"] == 1462.5 and s["reasons"] == ["sw_power_cap"]
    assert s["sm_mhz_bins"] == {"1400-1449": 1, "1450-1499": 2, "1500-1549": 1}
    assert s["sm_max_mhz"] == 2070 and s["sampler_period_ms"] == 50


def test_percentiles():
    p = bench.percentiles([5.0, 1.0, 2.0, 4.0, 3.0, 6.0, 7.0, 8.0, 9.0, 10.0])
    assert (p["min"], p["median"], p["p90"], p["mean"], p["n"]) == (1.0, 5.5, 9.0, 5.5, 10)


def test_datasheet_peaks_and_kernel_duration():
    # the percentage of the datasheet peak each config line carries: bf16 2250 TFLOP/s,
    # tf32 1100, exact fp32 (three tf32 products) 1100 / 3
    assert bench.datasheet_peak("bf16", "tensor") == 2250.0
    assert abs(bench.datasheet_peak("f32", "tensor") - 1100.0) < 1e-9
    assert abs(bench.datasheet_peak("f32", "tensor_x3") - 1100.0 / 3) < 1e-9
    # a step that is the kernel alone is timed over the region; with staging copies in the
    # step, the events around the kernel are used
    ms, how = bench.kernel_duration(10.0, 20, 20, 0.7)
    assert ms == 0.5 and "region" in how
    ms, how = bench.kernel_duration(10.0, 20, 60, 0.4)
    assert ms == 0.4 and "events" in how
