"""Host-side arithmetic of bench.py: the algorithmic work per step behind each
roofline fraction, and the lookup of committed ncu traffic. The expected
numbers are worked out here by hand from the workload's sizes."""
import json
from dataclasses import replace

import pytest

import bench
import workloads as wl

PEAKS = {"hbm_gbs": 6770.8, "bf16_tflops": 1898.2, "bf16_tflops_sustained": 1694.3}

# mlp_up: T = 16 x 1024 tokens, d_in 512, d_out 2048, K 8.
T, D_IN, D_OUT, K = 16384, 512, 2048, 8
ELEMENT_DRAWS = K * T * D_OUT           # 268,435,456
XU_PEAK = 16 * 152 * 2.07e9             # Box-Muller's transcendental pipe, per second


def test_workload_sizes_are_the_ones_worked_out_here():
    w = wl.MLP_UP
    assert (w.T, w.d_in, w.d_out, w.K) == (T, D_IN, D_OUT, K)
    assert w.element_draws == ELEMENT_DRAWS
    assert w.gemm_flops == 2 * T * D_IN * D_OUT


def test_gaussian_weighting_counts_two_xu_ops_per_element_draw():
    r = bench.roofline_for("weight", 0.125, [wl.MLP_UP], PEAKS)
    assert r["bound"] == "alu" and r["kernel"] == "weight"
    assert r["algorithmic_per_step"] == 2 * ELEMENT_DRAWS == 536870912
    assert r["peak"] * 1e9 == pytest.approx(XU_PEAK)
    assert r["frac"] == pytest.approx(536870912 / 0.125e-3 / XU_PEAK)


def test_antithetic_weighting_counts_half_the_noise_draws():
    r = bench.roofline_for("weight", 0.125, [wl.MLP_UP], PEAKS, antithetic=True)
    assert r["algorithmic_per_step"] == ELEMENT_DRAWS


def test_sign_weightings_count_alu_ops_and_issued_instructions():
    rad = replace(wl.MLP_UP, kind=0)
    packed = replace(wl.MLP_UP, kind=3)
    r = bench.roofline_for("weight", 0.1, [rad], PEAKS)
    assert r["algorithmic_per_step"] == 4 * ELEMENT_DRAWS
    assert r["peak"] * 1e9 == pytest.approx(64 * 152 * 2.07e9)
    p = bench.roofline_for("weight", 0.1, [packed], PEAKS)
    assert p["algorithmic_per_step"] == pytest.approx(3.25 * ELEMENT_DRAWS)
    assert p["peak"] * 1e9 == pytest.approx(128 * 152 * 2.07e9)


def test_contraction_counts_two_flop_per_multiply_add_against_sustained_peak():
    r = bench.roofline_for("gemm_tc", 0.04, [wl.MLP_UP], PEAKS)
    assert r["bound"] == "tensor"
    assert r["algorithmic_per_step"] == 34359738368
    assert r["frac"] == pytest.approx(34359738368 / 0.04e-3 / 1694.3e12)


def test_forward_counts_inputs_once_and_every_output_slice():
    # X and W read once, clean + 8 jittered slices written, all bf16.
    byts = 2 * (T * D_IN + D_OUT * D_IN + 9 * T * D_OUT)
    assert byts == 622854144
    r = bench.forward_roofline(0.125, T, D_IN, D_OUT, K, 1, 0, PEAKS)
    assert r["bound"] == "hbm" and r["algorithmic_per_step"] == byts
    assert r["frac"] == pytest.approx(byts / 0.125e-3 / 6770.8e9)
    # Gaussian: whichever of the XU and HBM fractions is larger bounds it.
    g = bench.forward_roofline(0.19, T, D_IN, D_OUT, K, 1, 1, PEAKS)
    xu = 2 * ELEMENT_DRAWS / 0.19e-3 / XU_PEAK
    hbm = byts / 0.19e-3 / 6770.8e9
    assert g["frac"] == pytest.approx(max(xu, hbm))
    assert g["bound"] == ("alu" if xu > hbm else "hbm")


def test_committed_traffic_is_read_only_while_its_sources_match(monkeypatch):
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        entries = json.load(f)
    for name, e in entries.items():
        kernel = "forward" if name.startswith("forward") else name
        entry = name if name.startswith("forward") else None
        got = bench.traffic_from_profiles(kernel, entry)
        if e["source_hash"] == bench.kernel_source_hash(kernel):
            assert got == e["dram_bytes_per_launch"]
        else:
            assert got is None
    assert bench.traffic_from_profiles("forward", "no_such_workload") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "0" * 16)
    for name in entries:
        kernel = "forward" if name.startswith("forward") else name
        assert bench.traffic_from_profiles(kernel, name if kernel == "forward" else None) is None
