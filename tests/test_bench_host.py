"""Host-side helpers of bench.py, on the CPU: clock-sample summary, the DRAM-traffic lookup in
the committed ncu summaries, and the L2 rule of the timed workloads."""

import pytest

import bench
from exact_tiled_attention_07_gb300.inputs import WORKLOADS


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.lines = lines
    return s


def _line(mhz, max_mhz=2070, power_cap="Not Active", thermal="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    return f"0, {mhz}, {max_mhz}, 900.0, 0x0, Not Active, Not Active, {thermal}, {power_cap}"


def test_clock_summary_keeps_the_timed_window():
    s = _sampler([(9.0, _line(1200)), (10.0, _line(2000)), (10.5, _line(2010, power_cap="Active")),
                  (11.0, _line(1990)), (20.0, _line(900, thermal="Active"))])
    got = s.summary(10.0, 11.0)
    assert got["samples"] == 3
    assert got["sm_mhz"] == 2000
    assert got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["sw_power_cap"]  # the thermal sample lies outside the window
    assert got["note"] == "samples inside the timed region"


def test_clock_summary_falls_back_to_every_sample_and_skips_malformed_lines():
    s = _sampler([(1.0, _line(1500, thermal="Active")), (2.0, "garbage"), (3.0, "0, [N/A], 2070, 1, 0, a, b, c, d")])
    got = s.summary(100.0, 101.0)
    assert got["samples"] == 1
    assert got["sm_mhz"] == 1500
    assert got["reasons"] == ["sw_thermal_slowdown"]
    assert got["note"].startswith("no sample fell inside")
    assert _sampler([]).summary(0.0, 1.0)["samples"] == 0


def test_profiled_traffic_only_for_the_current_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "x.md").write_text(
        "text\ntraffic: bwd_main causal_lm_bf16 1339600000 sources=abc\n"
        "traffic: fwd causal_lm_bf16 515500000 sources=old\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda: "abc")
    assert bench.profiled_traffic("bwd_main", "causal_lm_bf16") == 1339600000.0
    assert bench.profiled_traffic("bwd_main", "gpt2m_fp16") is None
    assert bench.profiled_traffic("fwd", "causal_lm_bf16") is None  # taken on other sources


def test_source_digest_is_stable():
    assert bench.source_digest() == bench.source_digest()
    assert len(bench.source_digest()) == 16


@pytest.mark.parametrize("name", ["causal_lm_bf16", "gpt2m_fp16", "long_causal_bf16", "hd256_bf16"])
def test_timed_workloads_have_inputs_larger_than_l2(name):
    # the bench flushes nothing between steps: each step's inputs must outgrow the 129 MB L2
    assert "larger than the 129 MB L2" in bench.l2_note(WORKLOADS[name])


def test_small_workload_is_reported_as_fitting_in_l2():
    assert "fit in L2" in bench.l2_note(WORKLOADS["tiny_fp32"])


def test_sm_clock_from_two_counter_readings():
    # SM 3: 2,070,000 cycles in 1 ms -> 2070 MHz; SM 5: 1,500,000 cycles in 1 ms -> 1500 MHz;
    # SM 9 appears only in the second reading and is ignored
    before = [(3, 10_000, 5_000_000), (5, 20_000, 5_000_100)]
    after = [(5, 1_520_000, 6_000_100), (3, 2_080_000, 6_000_000), (9, 1, 6_000_000)]
    got = sorted(bench.sm_clock_mhz(before, after))
    assert got == pytest.approx([1500.0, 2070.0])
    assert bench.sm_clock_mhz(before, []) == []


def test_peak_follows_the_length_of_the_timed_region():
    peaks = {"bf16_tflops": 1881.8, "bf16_tflops_sustained": 1707.9}
    assert bench.peak_for_region(peaks, 0.033) == (1881.8, "bf16_tflops (burst)")
    assert bench.peak_for_region(peaks, 5.0)[0] == 1707.9


def test_tensor_peak_at_clock():
    # 152 SMs x 8192 FLOP per clock at 2070 MHz
    assert bench.tensor_peak_at_clock(2070.0, 152) == pytest.approx(152 * 8192 * 2.07e9 / 1e12)
