"""Host-side logic of bench.py that the JSON line rests on, checked on the CPU: the
clock record's summary (median SM clock, throttle reasons that were active in any
sample), the per-step distribution, the committed DRAM-traffic figures (reported only
while the kernel sources match the hash they were taken on) and the algorithmic bytes
of the decode step."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from block_sparse_long_pool_gb300 import workloads as wl  # noqa: E402


def _sampler_with(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    (tmp_path / "clocks.csv").write_text("".join(l + "\n" for l in lines))
    s.proc = object()   # as if nvidia-smi had run
    return s


def test_clock_summary_takes_the_median_and_every_active_reason(tmp_path):
    # index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    s = _sampler_with(tmp_path, [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 950.3, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    ])
    out = s.summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_slowdowns_and_missing_samples(tmp_path):
    s = _sampler_with(tmp_path, [
        "0, 1200, 2070, 700.0, 0x0000000000000008, Active, Not Active, Active, Not Active",
    ])
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert _sampler_with(tmp_path, ["garbage"]).summary()["reasons"] == ["no samples"]
    none = bench.ClockSampler(0)
    assert none.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_step_distribution():
    d = bench.step_distribution([3.0, 1.0, 2.0, 5.0, 4.0])
    assert d == {"median": 3.0, "p10": 1.0, "p90": 5.0, "min": 1.0, "max": 5.0, "steps": 5}


@pytest.mark.parametrize("name,sources", [("decode_attn_128k_traffic.txt", bench.ATTN_SOURCES),
                                          ("decode_forecast_128k_traffic.txt", bench.FUSED_SOURCES),
                                          ("decode_forecast_128k_b1_traffic.txt", bench.FUSED_SOURCES)])
def test_traffic_figures_are_tied_to_the_kernel_sources(name, sources):
    """Each committed figure was taken on the current sources (its hash matches), so the
    bench reports it; any other hash gets None."""
    h = bench.kernel_source_hash(sources)
    traffic = bench.profiled_traffic(h, name)
    assert traffic is not None and traffic > 0
    assert bench.profiled_traffic("0" * 16, name) is None


def test_step_bytes_of_the_decode_workloads():
    """The algorithmic bytes the roofline divides: 67 selected 32 KB blocks per pair and
    layer, 2045 candidate compressed keys of 512 B per pair and layer (80 layers; layer
    0's selection is the extra launch, layer 79 selects nothing)."""
    for sh, pairs in ((wl.DECODE_128K, 64), (wl.DECODE_128K_B1, 8)):
        assert sh.pairs == pairs and sh.k_tot == 67 and bench.n_candidates(sh) == 2045
        step = bench.DecodeStep.algorithmic_bytes(type("S", (), {"sh": sh})())
        assert step == (80 * pairs * 67 * 32768, 80 * pairs * 2045 * 512)
    assert sum(bench.DecodeStep.algorithmic_bytes(type("S", (), {"sh": wl.DECODE_128K})())) == 16_601_579_520
