"""bench.py's roofline entry: which peak it divides by, and that a burst-length run of the
Mixtral-shape FFN at the rate measured on a B300 reads below 1 of its peak. CPU only."""
import importlib.util
import os

import pytest

from sparse_mixture_experts_70_b300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)

PEAKS = dict(bf16=1772.9, bf16_sustained=1366.0, hbm=6338.5, source="measured")


def _ffn_ms(w, tflops):
    return w.expert_flops() / (tflops * 1e12) * 1e3


def test_short_unthrottled_region_uses_the_burst_peak():
    # 20 steps of the Mixtral shape at 1572.7 TF/s (a 0.04 s region, no power cap)
    w = wl.WORKLOADS["mixtral"]
    r = bench.roofline(w, _ffn_ms(w, 1572.7), PEAKS, region_s=0.04, reasons=[])
    assert r["bound"] == "tensor" and r["peak"] == PEAKS["bf16"]
    assert r["frac"] == pytest.approx(1572.7 / 1772.9, rel=1e-6)
    assert r["frac"] <= 1.0
    assert r["frac_alt"] == pytest.approx(1572.7 / 1366.0, rel=1e-6)
    assert "burst" in r["peak_kind"] and "sustained" in r["frac_alt_kind"]


def test_short_region_under_the_power_cap_still_uses_the_burst_peak():
    w = wl.WORKLOADS["mixtral"]
    r = bench.roofline(w, _ffn_ms(w, 1300.0), PEAKS, region_s=0.5, reasons=["sw_power_cap"])
    assert r["peak"] == PEAKS["bf16"]


def test_long_power_capped_region_uses_the_sustained_peak():
    w = wl.WORKLOADS["mixtral"]
    r = bench.roofline(w, _ffn_ms(w, 1278.0), PEAKS, region_s=1.0,
                       reasons=["sw_power_cap"])
    assert r["peak"] == PEAKS["bf16_sustained"]
    assert r["frac"] == pytest.approx(1278.0 / 1366.0, rel=1e-6)
    assert r["frac_alt"] == pytest.approx(1278.0 / 1772.9, rel=1e-6)
    # a long region without the cap ran at burst clocks
    r2 = bench.roofline(w, _ffn_ms(w, 1278.0), PEAKS, region_s=5.0, reasons=[])
    assert r2["peak"] == PEAKS["bf16"]


@pytest.mark.parametrize("name,bound", [("mixtral", "tensor"), ("many_small", "tensor"),
                                        ("switch", "hbm"), ("decode", "hbm")])
def test_bound_follows_the_ridge_point(name, bound):
    w = wl.WORKLOADS[name]
    r = bench.roofline(w, 1.0, PEAKS, region_s=0.1, reasons=[])
    assert r["bound"] == bound
    ridge = PEAKS["bf16"] * 1e12 / (PEAKS["hbm"] * 1e9)
    assert (r["flop_per_byte"] >= ridge) == (bound == "tensor")
    if bound == "hbm":
        assert r["unit"] == "GB/s" and r["peak"] == PEAKS["hbm"]
        assert r["achieved"] == pytest.approx(w.ffn_bytes() / 1e-3 / 1e9)
    assert r["algorithmic_bytes_per_launch"] * r["launches_per_step"] == w.ffn_bytes()


def test_f32_layer_is_measured_against_the_ffma_rate():
    w = wl.WORKLOADS["micro"]
    alu = {"tflops": 70.0, "how": "FP32 FFMA, measured"}
    r = bench.roofline(w, _ffn_ms(w, 7.0), PEAKS, region_s=0.01, reasons=[], alu=alu)
    assert r["bound"] == "alu" and r["peak"] == 70.0
    assert r["frac"] == pytest.approx(0.1, rel=1e-6)


def test_traffic_is_labelled_with_its_source():
    w = wl.WORKLOADS["mixtral"]
    r = bench.roofline(w, 2.0, PEAKS, region_s=0.1, reasons=[],
                       traffic=bench.MEASURED_TRAFFIC["mixtral"])
    assert r["traffic"] == bench.MEASURED_TRAFFIC["mixtral"]["bytes"]
    assert "scaled" in r["traffic_source"]
    r = bench.roofline(w, 2.0, PEAKS, region_s=0.1, reasons=[], traffic=None)
    assert r["traffic"] is None and r["traffic_source"] is None


def test_backward_roofline_counts_twice_the_forward_flops():
    """The backward's algorithmic flops are the data and weight gradients of the expert GEMMs
    (twice the forward's); the Mixtral shape is tensor-bound, the decode shape HBM-bound (its
    weights read and its weight gradients written once)."""
    w = wl.WORKLOADS["mixtral"]
    ms = 2 * w.expert_flops() / 1000e12 * 1e3  # a backward at 1000 TF/s
    r = bench.backward_roofline(w, ms, PEAKS, region_s=0.5, reasons=[])
    assert r["bound"] == "tensor" and r["peak"] == PEAKS["bf16"]
    assert r["achieved"] == pytest.approx(1000.0, rel=1e-9)
    assert r["algorithmic_flops"] == 2 * w.expert_flops()
    d = wl.WORKLOADS["decode"]
    nbytes = 2 * d.weight_bytes() + 3 * d.T * d.d * 2
    r = bench.backward_roofline(d, nbytes / 5000e9 * 1e3, PEAKS, region_s=0.5, reasons=[])
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(5000.0, rel=1e-9)
    assert r["frac"] == pytest.approx(5000.0 / PEAKS["hbm"], rel=1e-9)


def test_power_capped_region_with_low_clocks_uses_the_sustained_peak():
    """A region shorter than a second but running under the power cap with its median SM clock at
    most 0.8 of the maximum is in the regime the sustained peak was measured in; with the clock
    near its maximum the burst peak stays."""
    w = wl.WORKLOADS["mixtral"]
    low = {"sm_mhz": 1218.5, "sm_max_mhz": 2032.0}
    r = bench.roofline(w, _ffn_ms(w, 1289.0), PEAKS, region_s=0.94, reasons=["sw_power_cap"],
                       clocks=low)
    assert r["peak"] == PEAKS["bf16_sustained"] and "sustained" in r["peak_kind"]
    assert r["frac_alt"] == pytest.approx(1289.0 / PEAKS["bf16"], rel=1e-6)
    high = {"sm_mhz": 1961.0, "sm_max_mhz": 2032.0}
    r = bench.roofline(w, _ffn_ms(w, 1289.0), PEAKS, region_s=0.94, reasons=["sw_power_cap"],
                       clocks=high)
    assert r["peak"] == PEAKS["bf16"]
    # low clocks without the power cap (a lock left by someone else) are not the sustained regime
    r = bench.roofline(w, _ffn_ms(w, 1289.0), PEAKS, region_s=0.94, reasons=[], clocks=low)
    assert r["peak"] == PEAKS["bf16"]
