"""Host logic of bench.py: launch counting, the recorded-traffic lookup and
its source hash, the peak figures and the clock summary (no GPU)."""
import json
import re

import pytest

import bench


def _call(name, nargs=13, x_perm=None):
    a = [None] * nargs
    if nargs > 10:
        a[10] = x_perm
    return (name, None, tuple(a))


def test_call_launches_counts_the_row_gather_only_when_it_runs():
    assert bench.call_launches(_call("moe_permute", x_perm=None)) == 1
    assert bench.call_launches(_call("moe_permute", x_perm=object())) == 2
    assert bench.call_launches(_call("moe_permute_ws", 15, x_perm=None)) == 3
    assert bench.call_launches(_call("moe_permute_ws", 15, x_perm=object())) == 4
    assert bench.call_launches(_call("moe_route")) == 2
    assert bench.call_launches(_call("moe_expert_swiglu_fused")) == 1
    assert bench.call_launches(_call("moe_combine_weighted")) == 1
    with pytest.raises(KeyError):
        bench.call_launches(_call("not_a_boundary_call"))


def test_committed_traffic_figures_match_the_committed_sources():
    """Every DRAM-traffic figure in profiles/traffic.json names the hash of
    the kernel sources it was captured on; the bench uses a figure only while
    that hash is current, so a committed figure must be current."""
    d = json.load(open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")))
    n = 0
    for kernel, entries in d.items():
        if kernel.startswith("_"):
            continue
        sha = bench.kernel_source_sha(kernel)
        assert re.fullmatch(r"[0-9a-f]{16}", sha)
        for workload, ent in entries.items():
            assert ent["src_sha"] == sha, (kernel, workload)
            assert ent["dram_bytes_per_unit"] > 0
            n += 1
    assert n >= 1


def test_recorded_traffic_scales_and_refuses_stale_or_unknown(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"fused": {"w": {"dram_bytes_per_unit": 1000, "src_sha": "0123456789abcdef"}}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda k: "0123456789abcdef")
    assert bench.recorded_traffic("fused", "w", 42.5) == 42500
    assert bench.recorded_traffic("fused", "other", 1) is None
    assert bench.recorded_traffic("gateup", "w", 1) is None
    monkeypatch.setattr(bench, "kernel_source_sha", lambda k: "ffffffffffffffff")
    assert bench.recorded_traffic("fused", "w", 1) is None
    (tmp_path / "profiles" / "traffic.json").write_text("{not json")
    assert bench.recorded_traffic("fused", "w", 1) is None
    (tmp_path / "profiles" / "traffic.json").unlink()
    assert bench.recorded_traffic("fused", "w", 1) is None


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.peaks()
    assert p["source"] == "fallback"
    assert p["hbm_gbs"] == bench.FALLBACK_HBM_GBS and p["bf16_tflops"] == bench.FALLBACK_BF16_TFLOPS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6000, "bf16_tflops": 1800}))
    p = bench.peaks()
    assert p == {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1800.0, "source": "measured"}
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6000, "bf16_tflops": 1800, "bf16_tflops_sustained": 1700}))
    assert bench.peaks()["bf16_tflops_sustained"] == 1700.0


def _sampler(samples):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = samples
    s.proc = None
    return s


def _row(sm, power, hw="Not Active", thermal="Not Active", sw_thermal="Not Active", cap="Not Active"):
    return [str(sm), "2070", str(power), "0x0", hw, thermal, sw_thermal, cap]


def test_clock_summary_takes_the_timed_window_and_names_active_reasons():
    s = _sampler([(0.5, _row(1000, 100)), (1.0, _row(2070, 700, cap="Active")), (1.5, _row(2000, 800)),
                  (2.0, _row(2070, 750)), (3.0, _row(500, 100, thermal="Active"))])
    c = s.summary(1.0, 2.0)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    assert c["power_w_max"] == 800.0
    c = s.summary(2.5, 3.5)
    assert c["reasons"] == ["hw_thermal_slowdown"] and c["sm_mhz"] == 500.0
    # no sample inside the window: every sample counts
    assert s.summary(10.0, 11.0)["samples"] == 5
    assert _sampler([]).summary(0.0, 1.0) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                                               "samples": 0}
