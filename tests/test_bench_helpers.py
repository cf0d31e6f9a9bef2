"""Host-side helpers of bench.py on CPU: the algorithmic byte counts the
roofline divides by, the percentile, the peaks and traffic records, the
clock-sample summary that decides whether a timed run is kept, and the
attention kernel label (the launchers' dispatch rule)."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_full_workload():
    # 256 queries x 4 heads x 128 fp32, 65,536 fp32 summary keys of 128,
    # 256 x 65,536 fp32 scores written once and read once, 256 x 512 int32 ids.
    a = bench.algorithmic(256, 65536, 512)
    q, keys, scores, ids = 524_288, 33_554_432, 67_108_864, 524_288
    assert a["score_bytes"] == q + keys + scores
    assert a["topk_bytes"] == scores + ids
    assert a["step_bytes"] == q + keys + 2 * scores + ids == 168_820_736
    # one query-block score: 4 heads x 128 multiply-adds = 1,024 flops; the
    # head-summed form (sum the heads first, one 128-long dot) = 256 flops.
    assert a["flops_per_head_form"] == 1024 * 256 * 65536
    assert a["flops_head_summed"] == 256 * 256 * 65536


def test_algorithmic_bytes_scale_linearly():
    a1 = bench.algorithmic(1, 4, 1)
    assert a1["step_bytes"] == 2048 + 2048 + 2 * 16 + 4
    a2 = bench.algorithmic(2, 4, 1)
    assert a2["topk_bytes"] == 2 * a1["topk_bytes"]


def test_step_floor_at_measured_peak():
    # the floor the headline fraction is taken against: 168.82 MB at the measured copy rate
    peaks = bench.load_peaks()
    floor_us = bench.algorithmic(256, 65536, 512)["step_bytes"] / (peaks["hbm_gbs"] * 1e3)
    assert 15.0 < floor_us < 40.0


def test_pct_nearest_rank():
    xs = [5.0, 1.0, 4.0, 2.0, 3.0]
    assert bench.pct(xs, 0) == 1.0
    assert bench.pct(xs, 50) == 3.0
    assert bench.pct(xs, 100) == 5.0
    assert bench.pct(xs, 25) == 2.0
    assert bench.pct([7.0], 90) == 7.0
    assert bench.pct(xs, 150) == 5.0 and bench.pct(xs, -10) == 1.0


def test_whole_job_rate_counts_every_rank():
    # 2 ranks x 1e6 units in a 1 ms step (max over ranks) -> 2e9 units/s
    assert bench.whole_job_rate(2, 1_000_000, 1.0) == pytest.approx(2e9)
    assert bench.whole_job_rate(1, 256 * 65536, 41.0e-3) == pytest.approx(256 * 65536 / 41.0e-6)


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_load_peaks_fields():
    p = bench.load_peaks()
    assert p["source"] in ("measured", "fallback")
    for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained", "sm_max_mhz"):
        assert p[key] > 0
    assert p["bf16_tflops_sustained"] <= p["bf16_tflops"] * 1.05


def test_recorded_traffic_matches_source_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "csrc"
    prof = tmp_path / "profiles"
    csrc.mkdir()
    prof.mkdir()
    (csrc / "k.cu").write_bytes(b"__global__ void k() {}\n")
    sha = hashlib.sha256(b"__global__ void k() {}\n").hexdigest()[:16]
    (prof / "dram_traffic.txt").write_text(
        f"kernel=k source_sha=0000000000000000 dram_bytes_per_launch=1\n"
        f"kernel=other source_sha={sha} dram_bytes_per_launch=2\n"
        f"kernel=k source_sha={sha} dram_bytes_per_launch=12345 workload=w\n")
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    monkeypatch.setattr(bench, "PROFILES", str(prof))
    assert bench.recorded_traffic("k", "k.cu") == 12345.0
    # a changed source invalidates the record
    (csrc / "k.cu").write_bytes(b"__global__ void k() { }\n")
    assert bench.recorded_traffic("k", "k.cu") is None
    assert bench.recorded_traffic("absent", "k.cu") is None


def test_recorded_traffic_committed_records_parse():
    # every committed record names a kernel, a 16-hex source hash and a byte count
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        pytest.skip("no traffic records")
    import re
    for line in open(p):
        if not line.strip():
            continue
        m = dict(re.findall(r"(\w+)=(\S+)", line))
        assert m["kernel"] and re.fullmatch(r"[0-9a-f]{16}", m["source_sha"])
        assert int(m["dram_bytes_per_launch"]) > 0


def _row(sm, smax, active="0x0000000000000000", hw="Not Active", hwt="Not Active", swt="Not Active",
         cap="Not Active", idx="0", power="900.00"):
    return ", ".join([idx, str(sm), str(smax), power, active, hw, hwt, swt, cap])


def test_clock_summary_median_and_reasons():
    lines = ["", "garbage line", _row(1900, 2070), _row(1950, 2070, cap="Active"), _row(2000, 2070)]
    s = bench.ClockSampler.summarise(lines)
    assert s["sm_mhz"] == 1950.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3


def test_clock_summary_flags_thermal_and_skips_na():
    lines = [_row("[N/A]", "[N/A]"), _row(1200, 2070, hwt="Active"), _row(1300, 2070, hw="Active")]
    s = bench.ClockSampler.summarise(lines)
    assert s["sm_mhz"] == 1250.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_clock_summary_empty_and_all_na():
    assert bench.ClockSampler.summarise([]) is None
    s = bench.ClockSampler.summarise([_row("[N/A]", "[N/A]")])
    assert s["sm_mhz"] is None and s["sm_max_mhz"] is None and s["samples"] == 1


def test_attn_kernel_label_follows_the_dispatch():
    # 152 SMs: clusters of 4 up to 38 queries, pairs up to 76, tensor cores beyond
    sms = 152
    assert bench.attn_kernel_label(1, sms).startswith("attn_kernel (CUDA cores, clusters of 4")
    assert bench.attn_kernel_label(38, sms).startswith("attn_kernel (CUDA cores, clusters of 4")
    assert bench.attn_kernel_label(39, sms).startswith("attn_kernel (CUDA cores, clusters of 2")
    assert bench.attn_kernel_label(76, sms).startswith("attn_kernel (CUDA cores, clusters of 2")
    assert "16-warp CTAs, 1 per SM" in bench.attn_kernel_label(77, sms)
    assert "16-warp CTAs, 1 per SM" in bench.attn_kernel_label(152, sms)
    assert "8-warp CTAs, 2 per SM" in bench.attn_kernel_label(153, sms)
    assert "8-warp CTAs, 2 per SM" in bench.attn_kernel_label(304, sms)
    assert "4-warp CTAs, 4 per SM" in bench.attn_kernel_label(305, sms)
