"""Host-side logic of bench.py: roofline denominators and byte accounting,
clock-sample parsing, and the rule that committed DRAM traffic is reported
only while the kernel's source still matches the digest it was taken on."""
import json
import os
import pathlib
import shutil

import pytest

import bench

REPO = bench.ROOT


@pytest.fixture
def scratch():
    """A scratch directory inside the repository's (git-ignored) pytest cache."""
    d = pathlib.Path(REPO) / ".pytest_cache" / "bench_host_scratch"
    shutil.rmtree(d, ignore_errors=True)
    d.mkdir(parents=True)
    yield d
    shutil.rmtree(d, ignore_errors=True)


def test_algorithmic_and_layout_bytes_closed_forms():
    # q4_K 4096 x 4096 at T = 512: 0.5625 B/weight, q8_1 1.125 B/activation, f32 Y
    assert bench.algorithmic_bytes("q4_K", 512, 4096, 4096) == 9437184 + 2359296 + 8388608
    # the layout reads the exact f16 hi/lo planes (4 B) plus scale words (0.125 B)
    assert bench.layout_bytes("q4_K", 512, 4096, 4096, 4) == 9437184 + 8650752 + 8388608
    # q6_K: 210 bytes per 256 weights
    assert bench.algorithmic_bytes("q6_K", 1, 4096, 4096) == 4096 * 16 * 210 + 4608 + 16384


def test_choose_peak_burst_only_at_max_clock_without_reasons():
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    at_max = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.choose_peak(peaks, at_max)[0] == 1900.0
    capped = dict(at_max, reasons=["sw_power_cap"])
    assert bench.choose_peak(peaks, capped)[0] == 1700.0
    low = {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.choose_peak(peaks, low)[0] == 1700.0
    assert bench.choose_peak(peaks, None)[0] == 1700.0
    # no sustained figure recorded: the burst one stands in
    assert bench.choose_peak({"bf16_tflops": 1900.0}, low)[0] == 1900.0


def test_job_throughput_is_all_ranks_over_the_slowest_time():
    # 100 GMAC per rank-step, 10 steps, 4 ranks, 2 ms -> 2000 TMAC/s
    assert bench.job_tmacs(100e9, 10, 4, 2.0) == pytest.approx(2000.0)


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_parses_samples_and_reasons(scratch):
    s = bench.ClockSampler(0)
    s.path = str(scratch / "clocks.csv")
    with open(s.path, "w") as fh:
        fh.write("0, 2070, 2070, 500.1, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        fh.write("0, 2070, 2070, 610.4, 0x4, Not Active, Not Active, Not Active, Active\n")
        fh.write("0, 1980, 2070, 605.0, 0x4, Not Active, Not Active, Not Active, Active\n")
        fh.write("garbage line\n")
    s.fh = open(os.devnull, "w")
    s.proc = _DoneProc()
    clk = s.stop()
    assert clk["samples"] == 3
    assert clk["sm_mhz"] == 2070.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["sw_power_cap"]
    assert clk["power_w_max"] == pytest.approx(610.4)
    assert not os.path.exists(s.path)


def test_clock_sampler_without_nvidia_smi_reports_no_clocks():
    s = bench.ClockSampler(0)
    s.proc = None
    clk = s.stop()
    assert clk["sm_mhz"] is None and clk["samples"] == 0


def test_traffic_reported_only_for_the_recorded_source(scratch, monkeypatch):
    root = scratch / "repo"
    csrc = root / "quantized_prefill_gemm_mmq_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (root / "profiles").mkdir()
    src = os.path.join(REPO, "quantized_prefill_gemm_mmq_gb300", "csrc")
    rec = json.load(open(os.path.join(REPO, "profiles", "traffic.json")))["mmq_q4K_sb_kernel"]
    for name in [rec["source"]] + rec["headers"]:
        shutil.copy(os.path.join(src, name), csrc / name)
    shutil.copy(os.path.join(REPO, "profiles", "traffic.json"), root / "profiles" / "traffic.json")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.traffic_bytes("mmq_q4K_sb_kernel") == rec["dram_bytes_per_launch"]
    # any change inside the kernel's source region invalidates the counters
    path = csrc / rec["source"]
    text = path.read_text()
    a = text.index(rec["region_begin"]) + len(rec["region_begin"])
    path.write_text(text[:a] + "\n// edited\n" + text[a:])
    assert bench.traffic_bytes("mmq_q4K_sb_kernel") is None
    # so does a change to one of the headers it is built from
    path.write_text(text)
    assert bench.traffic_bytes("mmq_q4K_sb_kernel") == rec["dram_bytes_per_launch"]
    hdr = csrc / rec["headers"][0]
    hdr.write_text(hdr.read_text() + "\n")
    assert bench.traffic_bytes("mmq_q4K_sb_kernel") is None
    assert bench.traffic_bytes("no_such_kernel") is None
