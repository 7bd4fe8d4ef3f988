"""Host-side pieces of bench.py that need no GPU: the clock record that decides
whether a run is rejected, the choice of the dominant kernel and the launch
count per call, and the lookup of profiled DRAM traffic."""
import bench


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.lines = lines
    return s.summary()


def test_clock_summary_median_and_reasons():
    lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1210.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = _sampler(lines)
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]           # kept and noted, not a rejection


def test_clock_summary_flags_thermal_and_skips_garbage():
    lines = [
        "0, 1800, 2070, 1390.0, 0x40, Not Active, Active, Not Active, Not Active",
        "not a sample",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1900, 2070, 1300.0, 0x20, Active, Not Active, Active, Not Active",
    ]
    s = _sampler(lines)
    assert s["samples"] == 2 and s["sm_mhz"] == 1850.0
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    s = _sampler([])
    assert s["samples"] == 0 and s["reasons"] == ["unavailable"] and s["sm_mhz"] is None


def test_dominant_kernel_and_launches_per_call():
    assert bench.dominant_kernel("nucleus_batch") == bench.KERNEL_NAME
    assert bench.launches_per_call("nucleus_batch") == 3    # greedy, keyhist, cluster
    assert bench.dominant_kernel("greedy") == bench.GREEDY_KERNEL
    assert bench.launches_per_call("greedy") == 1
    assert bench.dominant_kernel("mixed") == bench.FP32_KERNEL      # fp32 rows, B (K+1) = 3072
    assert bench.launches_per_call("mixed") == 4    # order, greedy, fp32 streaming, cluster
    assert bench.dominant_kernel("mtp_decode") == bench.CLUSTER_KERNEL   # B (K+1) = 2 rows


def test_profiled_traffic_reads_only_a_matching_source_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda: "abc123")
    f = prof / f"{bench.KERNEL_NAME}_nucleus_batch.md"
    f.write_text("source_hash: abc123\ntraffic_bytes_per_launch: 179354368\n")
    assert bench.profiled_traffic("nucleus_batch") == 179354368.0
    f.write_text("source_hash: 999999\ntraffic_bytes_per_launch: 179354368\n")
    assert bench.profiled_traffic("nucleus_batch") is None       # stale: the kernel changed
    assert bench.profiled_traffic("greedy") is None              # no summary for it here
