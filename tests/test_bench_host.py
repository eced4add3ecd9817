"""Host-side logic of bench.py: the choice of the peak the roofline divides by,
the clock-scaled tensor-pipe ceiling, the nvidia-smi clock summary and the
comment-insensitive source hash that keys the recorded ncu traffic."""
import os
import threading

import pytest

import bench


def test_choose_peak_burst_for_short_or_full_clock_regions():
    pk = {"bf16_tflops": 1908.0, "bf16_tflops_sustained": 1728.7}
    # under a second: the burst figure whatever the clock
    assert bench.choose_peak(pk, {"sm_mhz": 1500.0, "sm_max_mhz": 2070.0}, 0.5) == (1908.0, "burst")
    # seconds long but at the maximum clock: still burst
    assert bench.choose_peak(pk, {"sm_mhz": 2062.0, "sm_max_mhz": 2070.0}, 5.0) == (1908.0, "burst")
    # seconds long and clock-capped: the sustained figure
    assert bench.choose_peak(pk, {"sm_mhz": 1450.0, "sm_max_mhz": 2070.0}, 5.0) == (1728.7,
                                                                                   "sustained")
    # no clock samples: burst only for a short region
    assert bench.choose_peak(pk, {"sm_mhz": None, "sm_max_mhz": None}, 5.0)[1] == "sustained"
    # a missing figure falls back to the documented fallback peaks
    assert bench.choose_peak({}, {}, 0.1)[0] == bench.FALLBACK_PEAKS["bf16_tflops"]


def test_clock_peak_is_the_dense_pipe_rate_at_the_sampled_clock():
    # 152 SMs x 8192 FLOP per clock x 2070 MHz
    assert bench.clock_peak_tflops(2070.0) == pytest.approx(152 * 8192 * 2070e6 / 1e12)
    assert bench.clock_peak_tflops(None) is None
    assert bench.clock_peak_tflops(0) is None


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.proc = _FakeProc()
    s.thread = threading.Thread(target=lambda: None)
    s.thread.start()
    s.lines = list(lines)
    return s


def test_clock_summary_keeps_samples_inside_the_region():
    t0 = bench.ClockSampler._ts("2026/12/03 10:00:00.000")
    lines = [
        # before the region: ignored even though it reports a thermal slowdown
        "2026/12/03 09:59:59.000, 0, 900, 2070, 300.0, 0x0, Not Active, Active, Not Active, Not Active",
        "2026/12/03 10:00:00.100, 0, 2055, 2070, 650.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/03 10:00:00.200, 0, 2070, 2070, 690.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/03 10:00:00.300, 0, 2040, 2070, 700.0, 0x4, Not Active, Not Active, Not Active, Active",
        "malformed line",
    ]
    c = _sampler(lines).stop(t0, t0 + 0.35)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2055.0  # median of 2055, 2070, 2040
    assert c["sm_max_mhz"] == 2070.0
    assert c["power_w_max"] == 700.0
    assert c["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_samples_says_so():
    t0 = bench.ClockSampler._ts("2026/12/03 10:00:00.000")
    lines = ["2026/12/03 11:00:00.000, 0, 2070, 2070, 500.0, 0x0, Not Active, Not Active, "
             "Not Active, Not Active"]
    c = _sampler(lines).stop(t0, t0 + 1.0)
    assert c["sm_mhz"] is None
    assert "no samples inside the timed region" in c["reasons"][0]


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    csrc = tmp_path / "mask_aware_exact_gb300" / "csrc"
    csrc.mkdir(parents=True)

    def write(code):
        (csrc / "k.cu").write_text(code)
        return bench.kernel_source_hash(("k.cu",))

    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = write("int f(int x) {\n  return x + 1;\n}\n")
    # comments and indentation alone keep the hash
    assert write("// a note\nint f(int x) {  // why\n    return x + 1;\n}\n\n") == base
    # a code change does not
    assert write("int f(int x) {\n  return x + 2;\n}\n") != base
    assert len(base) == 12 and all(ch in "0123456789abcdef" for ch in base)


def test_recorded_traffic_keys_name_real_kernels_and_workload():
    # every recorded ncu traffic figure is keyed by a kernel the step times,
    # a 12-hex-digit source hash and the headline workload
    for key, val in bench.NCU_TRAFFIC.items():
        kernel, h, workload = key.split("@")
        assert kernel in bench.KERNEL_NAMES
        assert len(h) == 12 and all(ch in "0123456789abcdef" for ch in h)
        assert workload == "document_b1h32n32768d128"
        assert val > 0
