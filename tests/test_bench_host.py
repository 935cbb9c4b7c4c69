"""Host-side arithmetic of bench.py: the algorithmic work per step behind each
roofline fraction, and the lookup of committed ncu traffic. The expected
numbers are worked out here by hand from the workload's sizes."""
import json
from dataclasses import replace

import pytest

import bench
import workloads as wl

# Pipe rates as the probe reports them: per clock and SM, with the SM count
# and the probe's clock. 15.5 XU ops/clk/SM at 2000 MHz on 150 SMs, and so on.
PIPES = {"sm_count": 150, "probe_sm_mhz": 2000.0,
         "per_clk_per_sm": {"xu": 15.5, "alu": 60.0, "issue": 120.0, "fma": 250.0}}
PEAKS = {"hbm_gbs": 6770.8, "bf16_tflops": 1898.2, "bf16_tflops_sustained": 1694.3,
         "pipes": PIPES}

# mlp_up: T = 16 x 1024 tokens, d_in 512, d_out 2048, K 8.
T, D_IN, D_OUT, K = 16384, 512, 2048, 8
ELEMENT_DRAWS = K * T * D_OUT           # 268,435,456
XU_PEAK = 15.5 * 150 * 2000e6           # Box-Muller's transcendental pipe, per second


def test_workload_sizes_are_the_ones_worked_out_here():
    w = wl.MLP_UP
    assert (w.T, w.d_in, w.d_out, w.K) == (T, D_IN, D_OUT, K)
    assert w.element_draws == ELEMENT_DRAWS
    assert w.gemm_flops == 2 * T * D_IN * D_OUT


def test_gaussian_weighting_counts_two_xu_ops_per_element_draw():
    r = bench.roofline_for("weight", 0.125, [wl.MLP_UP], PEAKS)
    assert r["bound"] == "alu" and r["kernel"] == "weight" and r["pipe"] == "xu"
    assert r["algorithmic_per_step"] == 2 * ELEMENT_DRAWS == 536870912
    assert r["peak"] * 1e9 == pytest.approx(XU_PEAK)
    assert r["frac"] == pytest.approx(536870912 / 0.125e-3 / XU_PEAK)
    assert r["peak_source"].startswith("measured")


def test_measured_peaks_scale_with_the_timed_regions_clock():
    # the same per-clock rate at 1035 MHz is half the rate at 2070 MHz
    lo = bench.roofline_for("weight", 0.125, [wl.MLP_UP], PEAKS, clock_mhz=1035.0)
    hi = bench.roofline_for("weight", 0.125, [wl.MLP_UP], PEAKS, clock_mhz=2070.0)
    assert lo["peak"] * 1e9 == pytest.approx(15.5 * 150 * 1035e6)
    assert hi["frac"] == pytest.approx(lo["frac"] / 2)


def test_without_a_probe_the_peaks_are_derived_and_say_so():
    bare = {k: v for k, v in PEAKS.items() if k != "pipes"}
    r = bench.roofline_for("weight", 0.125, [wl.MLP_UP], bare)
    assert r["peak"] * 1e9 == pytest.approx(16 * 152 * 2070e6)
    assert r["peak_source"].startswith("derived")


def test_antithetic_weighting_counts_half_the_noise_draws():
    r = bench.roofline_for("weight", 0.125, [wl.MLP_UP], PEAKS, antithetic=True)
    assert r["algorithmic_per_step"] == ELEMENT_DRAWS


def test_sign_weightings_count_alu_ops_and_issued_instructions():
    rad = replace(wl.MLP_UP, kind=0)
    packed = replace(wl.MLP_UP, kind=3)
    r = bench.roofline_for("weight", 0.1, [rad], PEAKS)
    assert r["algorithmic_per_step"] == 4 * ELEMENT_DRAWS and r["pipe"] == "alu"
    assert r["peak"] * 1e9 == pytest.approx(60 * 150 * 2000e6)
    p = bench.roofline_for("weight", 0.1, [packed], PEAKS)
    assert p["algorithmic_per_step"] == pytest.approx(3.25 * ELEMENT_DRAWS)
    assert p["peak"] * 1e9 == pytest.approx(120 * 150 * 2000e6) and p["pipe"] == "issue"


def test_contraction_counts_two_flop_per_multiply_add_against_burst_peak():
    r = bench.roofline_for("gemm_tc", 0.04, [wl.MLP_UP], PEAKS)
    assert r["bound"] == "tensor"
    assert r["algorithmic_per_step"] == 34359738368
    assert r["frac"] == pytest.approx(34359738368 / 0.04e-3 / 1898.2e12)
    assert r["frac_of_sustained"] == pytest.approx(34359738368 / 0.04e-3 / 1694.3e12)


def test_sweep_work_sums_the_48_sites():
    sites = bench.workload_sites("sweep")
    assert len(sites) == 48
    # per layer: 512->1536, 512->512, 512->2048, 2048->512 over 65,536 tokens, K 32
    per_layer_el = 32 * 65536 * (1536 + 512 + 2048 + 512)
    assert sum(w.element_draws for w in sites) == 12 * per_layer_el
    assert sum(w.token_draws for w in sites) == 48 * 32 * 65536
    # down is 2048 -> 512: d_in d_out = 512 * 2048, as for up
    per_layer_fl = 2 * 65536 * 512 * (1536 + 512 + 2048 + 2048)
    r = bench.roofline_for("gemm_tc", 4.0, sites, PEAKS)
    assert r["algorithmic_per_step"] == 12 * per_layer_fl
    kinds = [bench.site_kind(w) for w in sites[:4]]
    assert kinds == ["qkv", "o", "up", "down"]
    one = bench.workload_sites("sweep_down")
    assert len(one) == 1 and (one[0].d_in, one[0].d_out) == (2048, 512)


def test_reference_sample_fits_its_time_budget():
    # 1 ms per token per step, 23 steps, 150 s: 6521 tokens -> capped at 1024
    assert bench.reference_sample_tokens(1e-3, 20, 3) == 1024
    # 50 ms per token: 150 / (0.05 * 23) = 130.4 -> 128 (a multiple of 16)
    assert bench.reference_sample_tokens(0.05, 20, 3) == 128
    # never below 16 tokens
    assert bench.reference_sample_tokens(10.0, 2000, 20) == 16


def test_forward_counts_inputs_once_and_every_output_slice():
    # X and W read once, clean + 8 jittered slices written, all bf16.
    byts = 2 * (T * D_IN + D_OUT * D_IN + 9 * T * D_OUT)
    assert byts == 622854144
    r = bench.forward_roofline(0.125, T, D_IN, D_OUT, K, 1, 0, PEAKS)
    assert r["bound"] == "hbm" and r["algorithmic_per_step"] == byts
    assert r["frac"] == pytest.approx(byts / 0.125e-3 / 6770.8e9)
    # Gaussian: whichever of the XU and HBM fractions is larger bounds it.
    g = bench.forward_roofline(0.19, T, D_IN, D_OUT, K, 1, 1, PEAKS, clock_mhz=2000.0)
    xu = 2 * ELEMENT_DRAWS / 0.19e-3 / XU_PEAK
    hbm = byts / 0.19e-3 / 6770.8e9
    assert g["frac"] == pytest.approx(max(xu, hbm))
    assert g["bound"] == ("alu" if xu > hbm else "hbm")


def test_committed_traffic_is_read_only_while_its_sources_match(monkeypatch):
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    for name, e in entries.items():
        kernel, workload = name.split(":")
        got = bench.traffic_from_profiles(kernel, workload)
        if e["source_hash"] == bench.kernel_source_hash(kernel):
            assert got == e["dram_bytes_per_launch"]
        else:
            assert got is None
    assert bench.traffic_from_profiles("forward", "no_such_workload") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "0" * 16)
    for name in entries:
        assert bench.traffic_from_profiles(*name.split(":")) is None


def test_sweep_traffic_is_the_mean_over_its_launches(monkeypatch):
    per = {"sweep_qkv": 4.0, "sweep_o": 1.0, "sweep_up": 6.0, "sweep_down": 1.0}
    monkeypatch.setattr(bench, "traffic_from_profiles", lambda k, w: per.get(w))
    sites = bench.workload_sites("sweep")
    assert bench.traffic_for("weight", "sweep", sites) == pytest.approx(3.0)
    per["sweep_o"] = None
    assert bench.traffic_for("weight", "sweep", sites) is None


def test_one_sweep_layer_is_its_four_sites():
    layer = bench.workload_sites("sweep_layer")
    sweep = bench.workload_sites("sweep")
    assert [bench.site_kind(w) for w in layer] == ["qkv", "o", "up", "down"]
    assert [(w.d_in, w.d_out, w.T, w.K, w.gamma) for w in layer] == \
        [(w.d_in, w.d_out, w.T, w.K, w.gamma) for w in sweep[:4]]
