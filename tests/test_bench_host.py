"""Host logic of the benchmark, without a GPU: the clock-sample summary that gates a run, the
ncu traffic lookup that is used only while the committed summary describes the current kernel
source, and the whole-job throughput arithmetic."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _clocks(lines):
    c = bench.Clocks(0)
    c.out = "\n".join(lines)
    return c.summary()


def test_clock_summary_median_max_and_reasons():
    rows = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1399.0, 0x0000000000000008, Active, Not Active, Not Active, Active",
        "garbage line",
    ]
    s = _clocks(rows)
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert _clocks(["", "nothing here"]) is None


def test_profile_traffic_only_for_the_current_kernel_source(tmp_path, monkeypatch):
    h = hashlib.sha256()
    for f in ("lossless_bit_weight_gb300/csrc/w12_gemm.cu", "lossless_bit_weight_gb300/csrc/w12_internal.cuh"):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    cur = h.hexdigest()[:16]
    p = tmp_path / "summary.md"
    p.write_text(f"# x\n\n- kernel_source_sha256_16: {cur}\n- dram_bytes_per_launch_full_size: 137.5e6 (note)\n")
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(p))
    assert bench.profile_traffic() == 137.5e6
    p.write_text("- kernel_source_sha256_16: 0000000000000000\n- dram_bytes_per_launch_full_size: 137.5e6\n")
    assert bench.profile_traffic() is None
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(tmp_path / "missing.md"))
    assert bench.profile_traffic() is None


def test_job_throughput_counts_every_rank_over_the_slowest():
    # two ranks, 1 GB each, the slower one taking 250 ms: 8 GB/s for the job
    assert abs(bench.job_gbs(1e9, 2, 250.0) - 8.0) < 1e-12
    assert bench.max_over_ranks(3.5) == 3.5
