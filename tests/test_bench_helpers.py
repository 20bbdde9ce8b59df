"""Host-side helpers of bench.py (no GPU): the algorithmic byte count of the
timed workload, the recorded-traffic lookup and its scaling, the host-link
bound, and the host description in the CPU baseline."""
import hashlib
import os

import bench
from zero_sharded_mixed_zero1_gb300 import workloads as W


def test_algorithmic_bytes_of_the_timed_workload():
    # 1.3e9 real parameters at 2M + 26 bytes (M = 8), 768 padding elements at 24
    w = W.FLAT_1P3B
    assert bench.algorithmic_bytes(w.n, 768, w.M) == 1_300_000_000 * 42 + 768 * 24 == 54_600_018_432


def test_recorded_traffic_is_scaled_and_tied_to_the_source(tmp_path, monkeypatch):
    cur = hashlib.sha256(b"".join(open(f, "rb").read() for f in bench.KERNEL_SOURCES)).hexdigest()
    prof = tmp_path / "prof.md"
    prof.write_text(f"- source_sha256: {cur}\n- replicas: 8\n- dram_bytes_per_launch: 1100\n"
                    f"- algorithmic_bytes_per_launch: 1000\n")
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(prof))
    traffic, note = bench.recorded_traffic(8, 50_000)
    assert traffic == 55_000 and "ratio 1.1000" in note
    assert bench.recorded_traffic(4, 50_000) == (None, None)          # another replica count
    prof.write_text(prof.read_text().replace(cur, "0" * 64))
    assert bench.recorded_traffic(8, 50_000) == (None, None)          # another kernel source


def test_committed_traffic_profile_matches_the_sources():
    """The committed small-case capture was taken on the kernel sources as
    they stand, so the bench reports its traffic."""
    traffic, _ = bench.recorded_traffic(8, 54_600_018_432)
    assert traffic is not None and 0.98 < traffic / 54_600_018_432 < 1.02


def test_link_roofline_takes_the_slowest_direction():
    link = {"h2d_gbs": 200.0, "d2h_gbs": 100.0, "both_directions_gbs": 250.0}
    r = bench.link_roofline(link, 20e9, 2e9, 0.125)
    assert abs(r["bound_ms"] - 100.0) < 1e-9           # 20 GB at 200 GB/s
    assert abs(r["frac"] - 0.8) < 1e-12
    r = bench.link_roofline(link, 1e9, 20e9, 0.25)
    assert abs(r["bound_ms"] - 200.0) < 1e-9           # 20 GB out at 100 GB/s


def test_host_cpu_description():
    d = bench.host_cpu()
    assert d["host_cpu_count"] == os.cpu_count() and d["host_cpu_count"] >= 1
    assert isinstance(d["cpu_model"], str) and d["cpu_model"]
    assert d["machine"]
