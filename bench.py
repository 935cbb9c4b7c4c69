#!/usr/bin/env python
"""Benchmark of the Dust per-token weight-gradient estimator on GB300.

Default workload: the whole-model sweep, the largest configuration. One step =
48 dust_estimate_gW calls on one stream, one per linear site of a 12-layer
transformer shape (d_model 512, MLP 2048; per layer QKV 512 -> 1536 with
gamma 0.9, O 512 -> 512, up 512 -> 2048 and down 2048 -> 512 with gamma 0),
each over 64 x 1024 tokens with K = 32 Gaussian draws, sigma 1e-3, bf16 X:
centring, credit scan, noise regeneration + reward weighting and the
contraction to GW, with inputs resident in HBM. `--workload` selects one
layer instead (mlp_up, qkv, the 4096^2 layers, the toy fp32 layer) or the
jittered forward (forward_*).

Metric: token-draws/s = sum over sites of K * T / step time (whole job over
all ranks). Prints one JSON line (rank 0). `--impl reference` times the fp64
CPU oracle on a bounded sample of the same workload instead (rank 0 only).

Timing: W warm-up steps, then K timed steps, each bracketed by CUDA events on
the launching stream with a 256 MB L2 flush between steps (outside the
events); barrier + synchronize around the timed region; max over ranks.
A second, profiled pass of the same steps times every kernel with events
(dust_profile_*) for the roofline of the dominant kernel; the rooflines of
the issue-bound kernels use pipe rates measured on the device by the
library's probe kernels (dust_pipe_probe), scaled to the SM clock sampled
during the timed region.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Dust ĜW token-draws/s at 1 GB300; % tensor-pipe peak (ĝᵀX) and % HBM (noise)"
UNIT = "token-draws/s"
SMI_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default per workload: sweep 20, square layers 100, "
                        "qkv 300, the rest 2000)")
    p.add_argument("--warmup", type=int, default=None,
                   help="warm-up steps (default: sweep 3, the rest 20)")
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="target wall time of the CPU-oracle sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--flags", type=int, default=None,
                   help="extra dust_estimate_gW flags (e.g. force a path)")
    p.add_argument("--workload", default="sweep",
                   choices=["sweep", "mlp_up", "toy", "qkv", "square_r", "square_g",
                            "square_rp", "sweep_qkv", "sweep_o", "sweep_up", "sweep_down",
                            "sweep_layer", "forward_g", "forward_r", "forward_rp"],
                   help="sweep (the 48-site whole-model pass, the largest configuration) is "
                        "the headline; sweep_layer is one of its layers (4 sites, the same "
                        "multi-site call); forward_* time the jittered forward (8 draws + the "
                        "clean output) of the up-projection layer; the others are single "
                        "layers (sweep_*: one site of each of the sweep's four shapes)")
    p.add_argument("--no-pipe-probe", action="store_true",
                   help="skip the pipe-rate probes (rooflines then use derived peaks)")
    args = p.parse_args(argv)
    steps, warm = DEFAULT_STEPS.get(args.workload, (2000, 20))
    if args.steps is None:
        args.steps = steps
    if args.warmup is None:
        args.warmup = warm
    return args


# (timed steps, warm-up steps) per workload: about a second of timed work.
DEFAULT_STEPS = {"sweep": (20, 3), "sweep_layer": (200, 10), "square_r": (100, 10),
                 "square_g": (100, 10), "square_rp": (100, 10), "qkv": (300, 20)}


# --------------------------------------------------------------- ranks ----

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(units_per_rank: float, ms_total: float, steps: int, world: int, backend_sync):
    """Whole-job throughput from each rank's device time: the max over ranks
    of the timed-region duration, units summed over ranks. `backend_sync`
    maps a local float to its max over ranks (identity at world size 1)."""
    ms_max = backend_sync(ms_total)
    ms_per_step = ms_max / steps
    value = world * units_per_rank * steps / (ms_max / 1000.0)
    return value, ms_per_step


# -------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + SMI_QUERY,
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        self.t0 = time.time()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        self.t1 = time.time()
        time.sleep(0.1)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm, smax, reasons, n = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (self.t0 <= ts <= self.t1 + 0.05):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": n}


# ------------------------------------------------------------ workload ----

def make_inputs(w, dev):
    """X (bf16), delta (planted quadratic loss, built with the library's own
    noise kernel, untimed) and sequence offsets, all resident on `dev`."""
    import numpy as np
    import torch
    import token_perturbation_estimator_gb300 as dust
    import workloads as wl

    X = torch.from_numpy(wl.make_X(w)).to(dev)
    if w.x_dtype == "bf16":
        X = X.to(torch.bfloat16)
    dplant = torch.from_numpy(wl.make_dplant(w)).to(dev)
    eps = torch.from_numpy(wl.make_eps(w)).to(dev)
    a = torch.empty((1, w.T, w.d_out), dtype=torch.float32, device=dev)
    dot = torch.empty((w.K, w.T), dtype=torch.float64, device=dev)
    sq = torch.empty((w.K, w.T), dtype=torch.float64, device=dev)
    for k in range(w.K):
        dust.dust_noise(a, w.seed, w.kind, k, 1, w.T, w.d_out)
        dot[k] = (a[0].double() * dplant.double()).sum(dim=1)
        sq[k] = (a[0].double() ** 2).sum(dim=1)
    delta = (w.sigma * dot + w.curvature * 0.5 * w.sigma * w.sigma * sq + eps.double()).float()
    so = torch.from_numpy(wl.seq_offsets(w)).to(dev)
    del a, dplant
    return X, delta.contiguous(), so


WORKLOADS = {
    "mlp_up": "mlp_up_512to2048_T16384_K8_gaussian",
    "toy": "toy_fp32_64x64_T256_K4_rademacher",
    "qkv": "qkv_1024to3072_T16384_K16_gaussian_gamma0.9",
    "square_r": "square_4096_T32768_K64_rademacher",
    "square_g": "square_4096_T32768_K64_gaussian",
    "square_rp": "square_4096_T32768_K64_rademacher_packed",
    "sweep": "sweep_12x4_sites_T65536_K32_gaussian",
    "sweep_layer": "sweep_1x4_sites_T65536_K32_gaussian",
    "sweep_qkv": "sweep_site_qkv_512to1536_T65536_K32_gaussian_gamma0.9",
    "sweep_o": "sweep_site_o_512to512_T65536_K32_gaussian",
    "sweep_up": "sweep_site_up_512to2048_T65536_K32_gaussian",
    "sweep_down": "sweep_site_down_2048to512_T65536_K32_gaussian",
    "forward_g": "forward_mlp_up_512to2048_T16384_8draws+clean_gaussian",
    "forward_r": "forward_mlp_up_512to2048_T16384_8draws+clean_rademacher",
    "forward_rp": "forward_mlp_up_512to2048_T16384_8draws+clean_rademacher_packed",
}
FORWARD_KIND = {"forward_g": 1, "forward_r": 0, "forward_rp": 3}
FORWARD_METRIC = "Dust jittered-forward token-draws/s at 1 GB300 (y = XW^T once, y + sigma a per draw)"


SWEEP_KINDS = ("qkv", "o", "up", "down")  # order of a layer's sites in the sweep


def workload_sites(name):
    import workloads as wl
    if name == "sweep":
        return wl.sweep_sites()
    if name == "sweep_layer":
        return wl.sweep_sites()[:len(SWEEP_KINDS)]
    if name.startswith("sweep_"):
        return [wl.sweep_sites()[SWEEP_KINDS.index(name[len("sweep_"):])]]
    return [{"mlp_up": wl.MLP_UP, "toy": wl.TOY, "qkv": wl.QKV_DECAY, "square_r": wl.SQUARE_R,
             "square_g": wl.SQUARE_G, "square_rp": wl.SQUARE_RP}[name]]


def site_kind(w):
    """The sweep shape a site belongs to ("qkv", "o", "up", "down"), or None."""
    for k in SWEEP_KINDS:
        if w.name.endswith("_" + k) and w.name.startswith("sweep_"):
            return k
    return None


def make_inputs_fast(w, dev, site):
    """Device-generated inputs for the many-site sweep: X ~ N(0, 1) in bf16
    from a seeded device generator, loss changes with the planted
    construction's marginal distribution (values do not change the work)."""
    import torch
    import workloads as wl
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + site)
    X = torch.randn((w.T, w.d_in), generator=g, device=dev).to(torch.bfloat16)
    delta = torch.from_numpy(wl.marginal_delta(w)).to(dev)
    so = torch.from_numpy(wl.seq_offsets(w)).to(dev)
    return X, delta, so


# ---------------------------------------------------------- roofline -----

# Per-SM, per-clock unit counts from public tables: used only when no pipe
# rates were measured (the CPU tests, or --no-pipe-probe).
DERIVED_PER_CLK_SM = {"xu": 16.0, "alu": 64.0, "issue": 128.0, "fma": 256.0}
DERIVED_SM, DERIVED_MHZ = 152, 2070.0


def measure_pipe_peaks(dust, dev, stream, target_ms=20.0, reps=5):
    """Rates of the XU, ALU, FMA and issue pipes on this device from the
    library's probe kernels (dust_pipe_probe), timed with CUDA events on
    `stream`, with the SM clock sampled meanwhile. Returns per-clock, per-SM
    rates so that a roofline can be scaled to the clock of another region."""
    import torch
    sink = torch.empty(dust.dust_pipe_probe_threads(), dtype=torch.float32, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pipes = {"xu": dust.PIPE_XU, "alu": dust.PIPE_ALU, "fma": dust.PIPE_FMA,
             "issue": dust.PIPE_ISSUE}
    rate = {}

    def timed(pipe, steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ops = dust.dust_pipe_probe(pipe, steps, sink, stream)
        b.record(stream)
        b.synchronize()
        return ops, a.elapsed_time(b)

    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for name, pipe in pipes.items():
            timed(pipe, 64)
            ops, ms = timed(pipe, 512)
            steps = int(max(64, min(1 << 24, 512 * target_ms / max(ms, 1e-3))))
            runs = [timed(pipe, steps) for _ in range(reps)]
            rate[name] = statistics.median(o / (m * 1e-3) for o, m in runs)
    cs = clk.summary()
    mhz = cs["sm_mhz"] or cs["sm_max_mhz"] or DERIVED_MHZ
    return {"sm_count": sms, "probe_sm_mhz": mhz, "probe_clock_samples": cs["samples"],
            "rate_per_s": rate,
            "per_clk_per_sm": {k: v / (sms * mhz * 1e6) for k, v in rate.items()}}


def pipe_peak(peaks, pipe, clock_mhz=None):
    """(ops/s, source) for `pipe`: the measured per-clock, per-SM rate times
    the SM count times the SM clock of the timed region (the probe's own
    clock when none was sampled); derived from unit counts when no probe
    ran."""
    m = peaks.get("pipes")
    if m:
        mhz = clock_mhz or m["probe_sm_mhz"]
        v = m["per_clk_per_sm"][pipe] * m["sm_count"] * mhz * 1e6
        return v, ("measured: dust_pipe_probe %s rate %.3g ops/clk/SM at %.0f MHz on %d SMs, "
                   "scaled to %.0f MHz (of measured)"
                   % (pipe, m["per_clk_per_sm"][pipe], m["probe_sm_mhz"], m["sm_count"], mhz))
    v = DERIVED_PER_CLK_SM[pipe] * DERIVED_SM * DERIVED_MHZ * 1e6
    return v, ("derived: %g ops/clk/SM x %d SMs x %.0f MHz (no probe run)"
               % (DERIVED_PER_CLK_SM[pipe], DERIVED_SM, DERIVED_MHZ))


def roofline_for(stage, ms_per_step, sites, peaks, antithetic=False, clock_mhz=None):
    """Roofline of the dominant kernel family, from its CUDA-event time per
    step and the algorithmic work of one step (summed over the step's sites):
      weight / fused (Gaussian): 2 transcendental (XU) ops per element-draw
        (Box-Muller's log, sqrt, sin, cos per channel pair) -> bound "alu"
        against the measured XU rate (lg2/sqrt/sin/cos.approx);
      weight / fused (Rademacher): 4 integer-ALU-pipe ops per element-draw (the
        key xor, fmix32's xor-shift by 13 (shift + xor) and the sign merge into
        the reward; its two multiplies issue on the FMA pipe) -> bound "alu"
        against the measured ALU rate (shr + xor);
      weight (packed signs): bound by instruction issue (ncu: issue slots 92 %
        busy, ALU 65 %, FMA 56 %): per element-draw 3 issued instructions (the
        shift that brings the channel's bit to the sign position, the masked
        xor into the reward, the add) plus the word's ~8 (key xor, two
        multiplies, two xor-shifts) shared by 32 channels -> 3.25 lane
        instructions per element-draw against the measured issue rate;
      gemm_tc: 2 T d_in d_out FLOP -> bound "tensor" against the measured
        burst bf16 peak (the contraction runs for microseconds to a few
        milliseconds at a time, inside steps far shorter than the seconds-long
        loop behind the sustained figure, which is reported beside it);
      gemm_simt: same FLOP on FFMA -> "alu" against the measured FMA rate.
    With antithetic pairs the weighting kernel evaluates each base draw's
    noise once (K / 2 noise draws per token); the fused kernel still K."""
    s = ms_per_step / 1000.0
    el = float(sum(w.element_draws for w in sites))
    if antithetic and stage == "weight":
        el /= 2.0
    fl = float(sum(w.gemm_flops for w in sites))
    if stage in ("weight", "fused"):
        if sites[0].kind == 1:
            ops, pipe = 2.0 * el, "xu"
        elif sites[0].kind == 3:
            ops, pipe = 3.25 * el, "issue"
        else:
            ops, pipe = 4.0 * el, "alu"
        peak, src = pipe_peak(peaks, pipe, clock_mhz)
        ach = ops / s
        return {"bound": "alu", "pipe": pipe, "achieved": ach / 1e9, "peak": peak / 1e9,
                "unit": "Gop/s", "frac": ach / peak, "traffic": None, "kernel": stage,
                "algorithmic_per_step": ops, "peak_source": src}
    if stage == "gemm_tc":
        peak = peaks.get("bf16_tflops", 1898.2) * 1e12
        sus = peaks.get("bf16_tflops_sustained", 1694.3) * 1e12
        ach = fl / s
        return {"bound": "tensor", "achieved": ach / 1e12, "peak": peak / 1e12,
                "unit": "TFLOP/s", "frac": ach / peak, "frac_of_sustained": ach / sus,
                "traffic": None, "kernel": stage, "algorithmic_per_step": fl,
                "peak_source": "MEASURED_PEAKS.json bf16_tflops, burst (of measured)"}
    peak, src = pipe_peak(peaks, "fma", clock_mhz)
    ach = fl / s
    return {"bound": "alu", "pipe": "fma", "achieved": ach / 1e12, "peak": peak / 1e12,
            "unit": "TFLOP/s", "frac": ach / peak, "traffic": None, "kernel": stage,
            "algorithmic_per_step": fl, "peak_source": src}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "fallback": True}


def forward_roofline(ms, T, d_in, d_out, K, clean, kind, peaks, clock_mhz=None):
    """Roofline of one jittered forward launch (k_forward):
      algorithmic bytes = 2 (T d_in + d_out d_in + (clean + K) T d_out): X and
        W read once, every output slice written once (bf16);
      Gaussian: 2 XU ops per element-draw (K T d_out), as for the weighting
        kernel -> bound "alu" against the measured XU rate when that fraction
        is the larger one;
      signs: bound "hbm" against the measured copy bandwidth."""
    s = ms / 1000.0
    byts = 2.0 * (T * d_in + d_out * d_in + (clean + K) * T * d_out)
    hbm = peaks.get("hbm_gbs", 6800.0) * 1e9
    out = {"bound": "hbm", "achieved": byts / s / 1e9, "peak": hbm / 1e9, "unit": "GB/s",
           "frac": byts / s / hbm, "traffic": None, "kernel": "forward",
           "algorithmic_per_step": byts,
           "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)"}
    if kind == 1:
        ops = 2.0 * K * T * d_out
        peak, src = pipe_peak(peaks, "xu", clock_mhz)
        if ops / s / peak > out["frac"]:
            out = {"bound": "alu", "pipe": "xu", "achieved": ops / s / 1e9, "peak": peak / 1e9,
                   "unit": "Gop/s", "frac": ops / s / peak, "traffic": None,
                   "kernel": "forward", "algorithmic_per_step": ops,
                   "hbm_frac": byts / s / hbm, "peak_source": src}
    return out


KERNEL_SOURCES = {
    "weight": ["k_weight.cu", "noise.cuh", "internal.cuh"],
    "gemm_tc": ["k_gemm_tc.cu", "tc_common.cuh", "internal.cuh"],
    "fused": ["k_fused.cu", "noise.cuh", "tc_common.cuh", "internal.cuh"],
    "forward": ["k_forward.cu", "noise.cuh", "tc_common.cuh", "internal.cuh"],
}


def kernel_source_hash(kernel):
    import hashlib
    files = KERNEL_SOURCES.get(kernel)
    if not files:
        return None
    h = hashlib.sha256()
    for f in files:
        p = os.path.join(ROOT, "token_perturbation_estimator_gb300", "csrc", f)
        if not os.path.exists(p):
            return None
        with open(p, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel, workload):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from a
    committed ncu capture (profiles/traffic.json, key "kernel:workload"), if
    the kernel's sources are unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get("%s:%s" % (kernel, workload))
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


def traffic_for(kernel, workload, sites):
    """Per-launch DRAM traffic of `kernel` over a step: for the sweep (or one
    of its layers), the mean over its launches of the four site shapes'
    captured traffic (None unless all four are current)."""
    if workload not in ("sweep", "sweep_layer"):
        return traffic_from_profiles(kernel, workload)
    per = {k: traffic_from_profiles(kernel, "sweep_" + k) for k in SWEEP_KINDS}
    if any(v is None for v in per.values()):
        return None
    return sum(per[site_kind(w)] for w in sites) / len(sites)


# ------------------------------------------------------------- cpu leg ----

def cpu_oracle_rate(sites, target_s):
    """Time the fp64 oracle on a bounded sample of the workload: whole
    sequences of each site (all channels, all draws), grown until the sample
    takes about target_s."""
    import numpy as np
    import oracle
    import workloads as wl

    def run(w, nseq):
        T = nseq * w.seq_len
        so = (np.arange(nseq + 1) * w.seq_len).astype(np.int32)
        rng = np.random.default_rng(7)
        X = wl.to_bf16_exact(rng.standard_normal((T, w.d_in), dtype=np.float32)) \
            if w.x_dtype == "bf16" else rng.standard_normal((T, w.d_in), dtype=np.float32)
        dp = rng.standard_normal((T, w.d_out), dtype=np.float32)
        eps = (w.eps_std * rng.standard_normal((w.K, T))).astype(np.float32)
        delta = oracle.planted_delta(dp, w.seed, w.kind, 0, w.K, np.float32(w.sigma),
                                     w.curvature, eps).astype(np.float32)
        t0 = time.perf_counter()
        oracle.estimate_gW(X, delta, w.d_out, so, w.seed, w.kind, 0, np.float32(w.sigma),
                           np.float32(w.gamma), 1.0, oracle.CENTER)
        return time.perf_counter() - t0, T

    kinds = {}
    for w in sites:  # one representative per distinct shape
        kinds.setdefault((w.d_in, w.d_out, w.gamma), w)
    reps = list(kinds.values())
    t1 = sum(run(w, 1)[0] for w in reps)
    nseq = int(max(1, min(min(w.n_seq for w in reps), round(target_s / max(t1, 1e-3)))))
    tot_t, tot_u, desc = 0.0, 0, []
    for w in reps:
        t, T = run(w, nseq)
        tot_t += t
        tot_u += w.K * T
        desc.append("%d of %d sequences of %d->%d (%d tokens x %d draws)"
                    % (nseq, w.n_seq, w.d_in, w.d_out, T, w.K))
    return {"value": tot_u / tot_t, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "sample": "; ".join(desc) + "; %.1f s" % tot_t}


def stage_fractions(prof, prof_steps, sites, peaks, anti, clock_mhz):
    """The metric's named fractions over a step: the contraction against the
    tensor peak (burst; sustained beside it), the noise/weighting stage
    against HBM (its bytes: the loss changes or rewards read, g written) and
    against its binding pipe."""
    out = {}
    if "gemm_tc" in prof:
        g = roofline_for("gemm_tc", prof["gemm_tc"]["total_ms"] / prof_steps, sites, peaks)
        out["gemm_tc_tensor_frac"] = g["frac"]
        out["gemm_tc_tensor_frac_of_sustained"] = g["frac_of_sustained"]
        if "reduce" in prof:
            ms = (prof["gemm_tc"]["total_ms"] + prof["reduce"]["total_ms"]) / prof_steps
            out["gemm_tc_with_reduce_tensor_frac"] = roofline_for("gemm_tc", ms, sites,
                                                                  peaks)["frac"]
    if "weight" in prof:
        byts = float(sum(4 * w.K * w.T + (2 if w.x_dtype == "bf16" else 4) * w.T * w.d_out
                         for w in sites))
        ms_w = prof["weight"]["total_ms"] / prof_steps
        out["weight_hbm_frac"] = byts / (ms_w / 1000.0) / (peaks.get("hbm_gbs", 6800.0) * 1e9)
        r = roofline_for("weight", ms_w, sites, peaks, anti, clock_mhz)
        out["weight_%s_frac" % r["pipe"]] = r["frac"]
    return out


def site_kind_breakdown(dust, bundles, flags, stream, flush, peaks, anti, clock_mhz, reps=5):
    """Per distinct site shape of a multi-site step: one site of that shape
    run `reps` times with per-kernel events; its kernels' times, their share
    of the site's profiled time, and the stage fractions."""
    import torch
    groups = {}
    for b in bundles:
        w = b["w"]
        groups.setdefault((w.d_in, w.d_out, w.gamma), []).append(b)
    out = {}
    for (d_in, d_out, gamma), bs in groups.items():
        b = bs[0]
        w = b["w"]
        dust.dust_profile_enable(True)
        dust.dust_profile_read()
        for _ in range(reps):
            flush.zero_()
            dust.dust_estimate_gW(b["X"], b["delta"], w.d_out, b["so"], w.seed, w.kind, 0,
                                  w.sigma, w.gamma, 1.0, flags, gW=b["gW"], workspace=b["ws"],
                                  stream=stream)
        torch.cuda.synchronize()
        prof = {k: {"launches": v[0], "total_ms": v[1]} for k, v in
                dust.dust_profile_read().items()}
        dust.dust_profile_enable(False)
        tot = sum(v["total_ms"] for v in prof.values()) / reps
        out[site_kind(w) or "%dx%d" % (d_in, d_out)] = {
            "d_in": d_in, "d_out": d_out, "gamma": gamma, "sites": len(bs),
            "us_per_site": {k: 1000.0 * v["total_ms"] / reps for k, v in prof.items()},
            "profiled_us_per_site": 1000.0 * tot,
            "stage_fractions": stage_fractions(prof, reps, [w], peaks, anti, clock_mhz)}
    return out


def reference_sample_tokens(step_s_per_token, steps, warmup, budget_s=150.0, cap=1024):
    """Tokens per site per reference step: one whole sequence (up to `cap`)
    when the run fits `budget_s`, fewer (a multiple of 16, at least 16) when
    it would not."""
    n = budget_s / max(1e-9, step_s_per_token * (steps + warmup))
    return int(max(16, min(cap, (int(n) // 16) * 16)))


def run_reference(args):
    """The reference arm: the fp64 CPU oracle, as it stands, on the host cores,
    on a bounded sample of the same workload per step (for the sweep: the
    first tokens of one sequence of each of its four site shapes, all draws
    and all channels; a single layer: the first tokens of one sequence)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    import workloads as wl

    sites = workload_sites(args.workload)
    reps = {}
    for w in sites:  # one representative per distinct shape
        reps.setdefault((w.d_in, w.d_out, w.gamma), w)
    reps = list(reps.values())
    rng = np.random.default_rng(7)

    def inputs(w, T):
        X = rng.standard_normal((T, w.d_in), dtype=np.float32)
        if w.x_dtype == "bf16":
            X = wl.to_bf16_exact(X)
        dp = rng.standard_normal((T, w.d_out), dtype=np.float32)
        eps = (w.eps_std * rng.standard_normal((w.K, T))).astype(np.float32)
        delta = oracle.planted_delta(dp, w.seed, w.kind, 0, w.K, np.float32(w.sigma),
                                     w.curvature, eps).astype(np.float32)
        return X, delta, np.array([0, T], np.int32)

    def step_fn(T):
        data = [(w, inputs(w, T)) for w in reps]

        def step():
            for w, (X, delta, so) in data:
                oracle.estimate_gW(X, delta, w.d_out, so, w.seed, w.kind, 0,
                                   np.float32(w.sigma), np.float32(w.gamma), 1.0, oracle.CENTER)
        return step

    # size the sample from one 16-token step
    probe = step_fn(16)
    t0 = time.perf_counter()
    probe()
    per_token = (time.perf_counter() - t0) / 16
    T = reference_sample_tokens(per_token, args.steps, args.warmup,
                                cap=min(w.seq_len for w in reps))
    step = step_fn(T)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    units = sum(w.K * T for w in reps)
    value = units * args.steps / dt
    cores = oracle.num_threads()
    sample = ("per step: the first %d tokens of one sequence of each of %d site shape(s) (%s), "
              "all draws and channels" % (T, len(reps), ", ".join(
                  "%d->%d gamma %g" % (w.d_in, w.d_out, w.gamma) for w in reps)))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "sample_tokens_per_site": T,
                   "site_shapes": len(reps), "token_draws_per_step": units},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- gpu leg ----

def run_gb300(args):
    import numpy as np
    import torch

    rank, world, local = dist_env()
    from __graft_entry__ import build
    build()
    import token_perturbation_estimator_gb300 as dust
    import workloads as wl

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
        pg = tdist

    def max_over_ranks(x):
        if pg is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        return float(t.item())

    def barrier():
        if pg is not None:
            pg.barrier()

    sites = workload_sites(args.workload)
    flags = dust.CENTER | (args.flags or 0)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    if not args.no_pipe_probe:
        peaks["pipes"] = measure_pipe_peaks(dust, dev, stream)
    fast = args.workload.startswith("sweep")
    bundles = []
    for i, w in enumerate(sites):
        if fast:
            X, delta, so = make_inputs_fast(w, dev, i)
        else:
            X, delta, so = make_inputs(w, dev)
        xd = dust.BF16 if X.dtype == torch.bfloat16 else dust.F32
        ws = torch.empty(dust.dust_estimate_gW_workspace(w.T, w.d_in, w.d_out, w.K, xd, flags),
                         dtype=torch.uint8, device=dev)
        gW = torch.empty((w.d_out, w.d_in), dtype=torch.float32, device=dev)
        bundles.append({"w": w, "X": X, "delta": delta, "so": so, "ws": ws, "gW": gW,
                        "path": dust.dust_estimate_gW_path(w.T, w.d_in, w.d_out, w.K, xd, flags)})
    units = sum(w.token_draws for w in sites)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MB > L2
    multi = len(bundles) > 1
    if multi:
        assert len({w.kind for w in sites}) == 1, "one noise kind per multi-site call"
        site_arr = dust.SiteArray([{"X": b["X"], "delta": b["delta"], "seq_offsets": b["so"],
                                    "gW": b["gW"], "workspace": b["ws"], "seed": b["w"].seed,
                                    "sigma": b["w"].sigma, "gamma": b["w"].gamma}
                                   for b in bundles])

    def step_sequential():
        # one dust_estimate_gW per site on one stream: each kernel runs alone
        for b in bundles:
            w = b["w"]
            dust.dust_estimate_gW(b["X"], b["delta"], w.d_out, b["so"], w.seed, w.kind, 0,
                                  w.sigma, w.gamma, 1.0, flags, gW=b["gW"], workspace=b["ws"],
                                  stream=stream)

    def step():
        # the whole model's sites in one call (the library's compute lanes)
        if multi:
            dust.dust_estimate_gW_sites(site_arr, sites[0].kind, 0, 1.0, flags, stream=stream)
        else:
            step_sequential()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st = dust.dust_last_error()
    if st != dust.OK:
        raise RuntimeError("device status after warm-up: " + dust.status_string(st))

    # ---- headline timed region
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for k in range(args.steps):
            flush.zero_()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    value, ms_per_step = aggregate(units, ms_total, args.steps, world, max_over_ranks)
    clock_summary = clocks.summary()
    clock_mhz = clock_summary.get("sm_mhz")

    # ---- the same sites one after another on one stream (no overlap between
    # sites): the reference point for the multi-site call's lanes
    seq_ms = None
    if multi:
        n_seq = max(1, min(args.steps, 5))
        for _ in range(2):
            flush.zero_()
            step_sequential()
        torch.cuda.synchronize()
        ts = []
        for _ in range(n_seq):
            flush.zero_()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step_sequential()
            b_.record(stream)
            b_.synchronize()
            ts.append(a.elapsed_time(b_))
        seq_ms = statistics.median(ts)

    # ---- profiled pass for per-kernel times: the sites one after another on
    # one stream, so that each kernel's events time it alone (in the timed
    # multi-site step kernels of different sites overlap, and a kernel's
    # bracketing events would include the time it shares the SMs); as many
    # steps as the library's profile buffer holds (one step's launch count
    # measured first)
    dust.dust_profile_enable(True)
    dust.dust_profile_read()
    flush.zero_()
    step_sequential()
    torch.cuda.synchronize()
    per_step = sum(v[0] for v in dust.dust_profile_read().values())
    prof_steps = max(1, min(args.steps, 60000 // max(1, per_step)))
    for k in range(prof_steps):
        flush.zero_()
        step_sequential()
    torch.cuda.synchronize()
    prof = {k: {"launches": v[0], "total_ms": v[1]} for k, v in dust.dust_profile_read().items()}
    dust.dust_profile_enable(False)
    launches_per_step = sum(v["launches"] for v in prof.values()) / prof_steps
    top = max(prof.items(), key=lambda kv: kv[1]["total_ms"])
    anti = bool(flags & dust.ANTITHETIC)
    roof = roofline_for(top[0], top[1]["total_ms"] / prof_steps, sites, peaks, anti, clock_mhz)
    roof["launches_per_step"] = top[1]["launches"] / prof_steps
    roof["traffic"] = traffic_for(top[0], args.workload, sites)
    # the same kernel family's work against the whole timed step (for the
    # multi-site call: with the sites' overlap)
    roof["frac_of_step"] = roof["frac"] * (top[1]["total_ms"] / prof_steps) / ms_per_step
    tot_ms = sum(x["total_ms"] for x in prof.values())
    breakdown = {k: {"launches": v["launches"],
                     "ms_per_launch": v["total_ms"] / v["launches"],
                     "share": v["total_ms"] / tot_ms}
                 for k, v in prof.items()}
    stage_fracs = stage_fractions(prof, prof_steps, sites, peaks, anti, clock_mhz)
    per_kind = None
    if len(sites) > 1:
        per_kind = site_kind_breakdown(dust, bundles, flags, stream, flush, peaks, anti,
                                       clock_mhz)

    # ---- end to end through the host-buffer C ABI entry points: one
    # dust_estimate_gW_host call for a single layer, one
    # dust_estimate_gW_host_sites call for the whole sweep
    hosts = []
    for b in bundles:
        hosts.append({"Xh": b["X"].cpu().pin_memory(), "dh": b["delta"].cpu().pin_memory(),
                      "sh": b["so"].cpu().pin_memory(),
                      "gh": torch.empty(tuple(b["gW"].shape), dtype=torch.float32).pin_memory(),
                      "Xs": torch.empty_like(b["X"]), "ds": torch.empty_like(b["delta"]),
                      "ss": torch.empty_like(b["so"]), "gs": torch.empty_like(b["gW"])})
    host_sites = [{"X_host": h["Xh"], "X_dev": h["Xs"], "delta_host": h["dh"],
                   "delta_dev": h["ds"], "seq_host": h["sh"], "seq_dev": h["ss"],
                   "gW_host": h["gh"], "gW_dev": h["gs"], "workspace": b["ws"],
                   "seed": b["w"].seed, "sigma": b["w"].sigma, "gamma": b["w"].gamma}
                  for b, h in zip(bundles, hosts)]

    def e2e_step():
        # returns (host enqueue, wait for the stream) in seconds
        a = time.perf_counter()
        if len(bundles) > 1:
            dust.dust_estimate_gW_host_sites(host_sites, sites[0].kind, 0, 1.0, flags,
                                             stream=stream)
        else:
            b, h = bundles[0], hosts[0]
            w = b["w"]
            dust.dust_estimate_gW_host(h["Xh"], h["Xs"], h["dh"], h["ds"], h["sh"], h["ss"],
                                       h["gh"], h["gs"], w.d_out, w.seed, w.kind, 0, w.sigma,
                                       w.gamma, 1.0, flags, workspace=b["ws"], stream=stream)
        b_ = time.perf_counter()
        stream.synchronize()
        return b_ - a, time.perf_counter() - b_

    n_e2e = max(3, min(args.e2e_steps, args.steps)) if len(sites) > 1 else args.e2e_steps
    for _ in range(3):
        e2e_step()
    barrier()
    torch.cuda.synchronize()
    e2e_times, e2e_split = [], []
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        a = time.perf_counter()
        e2e_split.append(e2e_step())
        e2e_times.append(time.perf_counter() - a)
    e2e_s = max_over_ranks(time.perf_counter() - t0)
    e2e_value = world * units * n_e2e / e2e_s
    # The host link's rate for this step's inputs: every X copied host -> device
    # on one stream with nothing else running (the bound the inputs put on e2e).
    link = torch.cuda.Stream()
    la, lb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    la.record(link)
    with torch.cuda.stream(link):
        for h in hosts:
            h["Xs"].copy_(h["Xh"], non_blocking=True)
    lb.record(link)
    lb.synchronize()
    x_bytes = sum(h["Xh"].numel() * h["Xh"].element_size() for h in hosts)
    link_gbs = x_bytes / (la.elapsed_time(lb) * 1e-3) / 1e9
    h2d = sum(h["Xh"].numel() * h["Xh"].element_size() + h["dh"].numel() * 4 +
              h["sh"].numel() * 4 for h in hosts)
    d2h = sum(h["gh"].numel() * 4 for h in hosts)
    # the two results agree (same arguments, deterministic)
    for b, h in zip(bundles, hosts):
        if not torch.equal(h["gh"], b["gW"].cpu()):
            raise RuntimeError("host-buffer path disagrees with the device path")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_rate(sites, args.cpu_seconds)

    if rank == 0:
        w0 = sites[0]
        cfg = {"workload": WORKLOADS[args.workload], "sites": len(sites),
               "token_draws_per_step": units,
               "noise": {0: "rademacher", 1: "gaussian", 3: "rademacher_packed"}[w0.kind],
               "x_dtype": w0.x_dtype, "paths": sorted({b["path"] for b in bundles}),
               "parallelism": "replicas" if world > 1 else "single",
               "entry_point": "dust_estimate_gW_sites" if multi else "dust_estimate_gW",
               "l2": "flushed (256 MB write) between timed steps"}
        if len(sites) == 1:
            cfg.update({"d_in": w0.d_in, "d_out": w0.d_out, "T": w0.T, "n_seq": w0.n_seq,
                        "K": w0.K, "sigma": w0.sigma, "gamma": w0.gamma})
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w0.x_dtype == "bf16" else "f32", "data": "synthetic",
            "config": cfg,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": n_e2e,
                    "ms_per_step_min_median_max": [1000.0 * min(e2e_times),
                                                   1000.0 * statistics.median(e2e_times),
                                                   1000.0 * max(e2e_times)],
                    "x_h2d_link_gbs": link_gbs,
                    # every step, and the slowest step's host enqueue and wait (ms)
                    "ms_per_step_all": [round(1000.0 * t, 2) for t in e2e_times],
                    "slowest_step_enqueue_wait_ms": [
                        round(1000.0 * x, 2) for x in e2e_split[e2e_times.index(max(e2e_times))]],
                    "entry_point": "dust_estimate_gW_host_sites" if len(sites) > 1
                    else "dust_estimate_gW_host"},
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": clock_summary,
            "breakdown": breakdown,
            "stage_fractions": stage_fracs,
            "sites_by_shape": per_kind,
            "pipe_peaks": peaks.get("pipes"),
            "gw_updates_per_s": len(sites) * 1000.0 / ms_per_step,
            "profiled_ms_per_step": tot_ms / prof_steps,
            "profiled_steps": prof_steps,
            "profile_mode": "sites one after another on one stream" if multi else "the step",
            "sites_call": {"entry_point": "dust_estimate_gW_sites", "lanes": dust.dust_estimate_gW_sites_lanes(),
                           "sequential_ms_per_step": seq_ms} if multi else None,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


# ----------------------------------------------------- jittered forward ----

def forward_inputs():
    import workloads as wl
    w = wl.MLP_UP
    X = wl.to_bf16_exact(wl.make_X(w))
    W = wl.to_bf16_exact(wl.make_W(w))
    return w, X, W


def cpu_forward_rate(kind, target_s):
    """The fp64 oracle's jittered forward on a bounded sample: the first Ts
    tokens of the layer (all channels, all draws, the clean slice), Ts grown
    until the sample takes about target_s."""
    import numpy as np
    import oracle
    w, X, W = forward_inputs()

    def run(Ts):
        t0 = time.perf_counter()
        oracle.forward_jitter(X[:Ts], W, w.seed, kind, 0, w.K, w.sigma, clean=True)
        return time.perf_counter() - t0

    t1 = run(64)
    Ts = int(max(64, min(w.T, 64 * round(target_s / max(t1, 1e-3)))))
    dt = run(Ts)
    return {"value": w.K * Ts / dt, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "first %d of %d tokens, %d draws + clean, all %d channels; %.1f s"
                      % (Ts, w.T, w.K, w.d_out, dt)}


def run_forward_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w, X, W = forward_inputs()
    kind = FORWARD_KIND[args.workload]
    Ts = 128  # one token tile per step: the oracle's full path on it

    def step():
        oracle.forward_jitter(X[:Ts], W, w.seed, kind, 0, w.K, w.sigma, clean=True)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = w.K * Ts * args.steps / dt
    line = {
        "impl": "reference", "metric": FORWARD_METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "sample_tokens_per_step": Ts},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": "%d tokens per step, all draws and channels" % Ts},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_forward(args):
    """One step = one dust_forward_jitter call: y = X W^T of the MLP
    up-projection layer (16384 tokens, 512 -> 2048, bf16) and its 8 jittered
    outputs plus the clean one, all written to HBM."""
    import torch
    rank, world, local = dist_env()
    from __graft_entry__ import build
    build()
    import token_perturbation_estimator_gb300 as dust

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
        pg = tdist

    def max_over_ranks(x):
        if pg is None:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        return float(t.item())

    def barrier():
        if pg is not None:
            pg.barrier()

    kind = FORWARD_KIND[args.workload]
    w, Xn, Wn = forward_inputs()
    K, T = w.K, w.T
    X = torch.from_numpy(Xn).to(dev).to(torch.bfloat16)
    W = torch.from_numpy(Wn).to(dev).to(torch.bfloat16)
    Y = torch.empty((K + 1, T, w.d_out), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    units = K * T
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MB > L2

    def step():
        dust.dust_forward_jitter(X, W, w.seed, kind, 0, K, w.sigma, clean=True, Y=Y,
                                 stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st = dust.dust_last_error()
    if st != dust.OK:
        raise RuntimeError("device status after warm-up: " + dust.status_string(st))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for k in range(args.steps):
            flush.zero_()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    value, ms_per_step = aggregate(units, ms_total, args.steps, world, max_over_ranks)

    clock_summary = clocks.summary()
    dust.dust_profile_enable(True)
    dust.dust_profile_read()
    for k in range(args.steps):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    prof = dust.dust_profile_read()
    dust.dust_profile_enable(False)
    launches, fwd_ms = prof["forward"]
    peaks = load_peaks()
    if not args.no_pipe_probe:
        peaks["pipes"] = measure_pipe_peaks(dust, dev, stream)
    roof = forward_roofline(fwd_ms / launches, T, w.d_in, w.d_out, K, 1, kind, peaks,
                            clock_summary.get("sm_mhz"))
    roof["launches_per_step"] = launches / args.steps
    roof["traffic"] = traffic_from_profiles("forward", args.workload)

    # end to end: X and W from pinned host memory, every output slice back
    Xh, Wh = X.cpu().pin_memory(), W.cpu().pin_memory()
    Yh = torch.empty(tuple(Y.shape), dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        X.copy_(Xh, non_blocking=True)
        W.copy_(Wh, non_blocking=True)
        step()
        Yh.copy_(Y, non_blocking=True)
        stream.synchronize()

    n_e2e = max(3, min(args.e2e_steps, 50))
    for _ in range(3):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - t0)
    e2e_value = world * units * n_e2e / e2e_s
    if not torch.equal(Yh, Y.cpu()):
        raise RuntimeError("host copy of the outputs disagrees with the device")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_forward_rate(kind, args.cpu_seconds)
    if rank == 0:
        cfg = {"workload": WORKLOADS[args.workload], "d_in": w.d_in, "d_out": w.d_out, "T": T,
               "draws": K, "clean_slice": True, "sigma": w.sigma,
               "noise": {0: "rademacher", 1: "gaussian", 3: "rademacher_packed"}[kind],
               "x_dtype": "bf16", "y_dtype": "bf16",
               "parallelism": "replicas" if world > 1 else "single",
               "l2": "flushed (256 MB write) between timed steps"}
        line = {
            "metric": FORWARD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": cfg, "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": (Xh.numel() + Wh.numel()) * 2,
                    "d2h_bytes_per_step": Yh.numel() * 2},
            "gpu_launches": int(launches),
            "clocks": clock_summary,
            "pipe_peaks": peaks.get("pipes"),
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    forward = args.workload.startswith("forward_")
    if args.impl == "reference":
        return run_forward_reference(args) if forward else run_reference(args)
    return run_forward(args) if forward else run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
