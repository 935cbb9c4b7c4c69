"""Seeded synthetic workloads shared by the tests and the benchmark.

This module holds shapes and random inputs only: no hash, no noise, no step
of the estimator. Where an input needs the estimator's noise (the planted
loss changes), the caller computes the two per-(draw, token) reductions
<dplant_t, a_t> and |a_t|^2 with its own noise source and hands them to
`assemble_delta`.

Workloads follow the five synthetic configurations measured by this project:
a toy fp32 layer, an MLP up-projection, a fused QKV projection with credit
decay, a large square layer (Rademacher and Gaussian), and a 12-layer sweep
of 48 linear sites. Seeds: estimator 0, X 1, planted error 2, loss noise 3,
layer weight 4 (the jittered forward).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

RADEMACHER = 0
GAUSSIAN = 1
RADEMACHER_PACKED = 3  # 32 signs per hash word

SEED_EST, SEED_X, SEED_PLANT, SEED_EPS, SEED_W = 0, 1, 2, 3, 4


@dataclass(frozen=True)
class Workload:
    name: str
    d_in: int
    d_out: int
    n_seq: int
    seq_len: int
    K: int
    sigma: float
    gamma: float
    kind: int
    x_dtype: str          # "f32" or "bf16"
    curvature: float      # weight of the 0.5 sigma^2 |a|^2 term in delta
    eps_std: float = 1e-2  # std of the N(0, 1e-4) loss-noise term
    x_channel_scale: bool = False  # X[:, j] *= s_j, s_j ~ U(0.5, 2)
    seed: int = SEED_EST

    @property
    def T(self) -> int:
        return self.n_seq * self.seq_len

    @property
    def token_draws(self) -> int:
        return self.K * self.T

    @property
    def element_draws(self) -> int:
        return self.K * self.T * self.d_out

    @property
    def gemm_flops(self) -> int:
        return 2 * self.T * self.d_in * self.d_out

    def scaled(self, n_seq=None, seq_len=None, K=None, d_in=None, d_out=None):
        """A smaller copy with the same distributions (for the oracle)."""
        kw = {}
        if n_seq is not None:
            kw["n_seq"] = n_seq
        if seq_len is not None:
            kw["seq_len"] = seq_len
        if K is not None:
            kw["K"] = K
        if d_in is not None:
            kw["d_in"] = d_in
        if d_out is not None:
            kw["d_out"] = d_out
        return replace(self, name=self.name + "-small", **kw)


TOY = Workload("toy_fp32_64x64_T256_K4_rademacher", 64, 64, 2, 128, 4, 1e-2, 0.0,
               RADEMACHER, "f32", 0.0)
MLP_UP = Workload("mlp_up_512to2048_T16384_K8_gaussian", 512, 2048, 16, 1024, 8, 1e-3, 0.0,
                  GAUSSIAN, "bf16", 1.0)
QKV_DECAY = Workload("qkv_1024to3072_T16384_K16_gaussian_gamma0.9", 1024, 3072, 8, 2048, 16,
                     1e-3, 0.9, GAUSSIAN, "bf16", 1.0)
SQUARE_R = Workload("square_4096_T32768_K64_rademacher", 4096, 4096, 32, 1024, 64, 5e-4, 0.0,
                    RADEMACHER, "bf16", 1.0, x_channel_scale=True)
SQUARE_G = Workload("square_4096_T32768_K64_gaussian", 4096, 4096, 32, 1024, 64, 5e-4, 0.0,
                    GAUSSIAN, "bf16", 1.0, x_channel_scale=True)
# The square layer with packed signs (32 per hash word): same shapes and draws.
SQUARE_RP = Workload("square_4096_T32768_K64_rademacher_packed", 4096, 4096, 32, 1024, 64,
                     5e-4, 0.0, RADEMACHER_PACKED, "bf16", 1.0, x_channel_scale=True)


def sweep_sites():
    """The 12-layer transformer sweep: 48 sites, 64 x 1024 tokens, K=32."""
    sites = []
    for layer in range(12):
        for nm, d_in, d_out, gamma in (("qkv", 512, 1536, 0.9), ("o", 512, 512, 0.0),
                                       ("up", 512, 2048, 0.0), ("down", 2048, 512, 0.0)):
            sites.append(Workload("sweep_l%d_%s" % (layer, nm), d_in, d_out, 64, 1024, 32,
                                  1e-3, gamma, GAUSSIAN, "bf16", 1.0,
                                  seed=SEED_EST + len(sites)))
    return sites


CONFIGS = {w.name: w for w in (TOY, MLP_UP, QKV_DECAY, SQUARE_R, SQUARE_G, SQUARE_RP)}


def seq_offsets(w: Workload) -> np.ndarray:
    return (np.arange(w.n_seq + 1, dtype=np.int64) * w.seq_len).astype(np.int32)


def make_X(w: Workload, seed: int = SEED_X) -> np.ndarray:
    """X [T, d_in] as float32 (round it to bf16 with `to_bf16_exact`)."""
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((w.T, w.d_in), dtype=np.float32)
    if w.x_channel_scale:
        s = rng.uniform(0.5, 2.0, size=w.d_in).astype(np.float32)
        X *= s[None, :]
    return X


def make_W(w: Workload, seed: int = SEED_W) -> np.ndarray:
    """Layer weight W [d_out, d_in] ~ N(0, 1/d_in) as float32 (the jittered
    forward's second operand; round it to bf16 with `to_bf16_exact`)."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((w.d_out, w.d_in), dtype=np.float32)
            / np.float32(np.sqrt(w.d_in))).astype(np.float32)


def make_dplant(w: Workload, seed: int = SEED_PLANT) -> np.ndarray:
    """Planted output error delta_t ~ N(0, I), [T, d_out] float32."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((w.T, w.d_out), dtype=np.float32)


def make_eps(w: Workload, seed: int = SEED_EPS) -> np.ndarray:
    """Loss-noise term N(0, 1e-4) (variance 1e-4), [K, T] float32."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((w.K, w.T), dtype=np.float32) * w.eps_std).astype(np.float32)


def assemble_delta(w: Workload, dot: np.ndarray, sq: np.ndarray, eps: np.ndarray) -> np.ndarray:
    """delta[k, t] = sigma*dot + curvature*0.5*sigma^2*sq + eps, as float32."""
    d = (w.sigma * np.asarray(dot, np.float64)
         + w.curvature * 0.5 * w.sigma * w.sigma * np.asarray(sq, np.float64)
         + np.asarray(eps, np.float64))
    return d.astype(np.float32)


def marginal_delta(w: Workload, seed: int = SEED_EPS) -> np.ndarray:
    """Loss changes with the planted construction's marginal distribution but
    no coupling to the noise: mean curvature*0.5*sigma^2*d_out, variance
    sigma^2*d_out + eps_std^2. Used where only the arithmetic is under test."""
    rng = np.random.default_rng(seed + 1000)
    mean = w.curvature * 0.5 * w.sigma * w.sigma * w.d_out
    std = float(np.sqrt(w.sigma * w.sigma * w.d_out + w.eps_std * w.eps_std))
    return (mean + std * rng.standard_normal((w.K, w.T))).astype(np.float32)


def to_bf16_exact(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even) and return the values as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    r = ((u + rounding) >> 16) << 16
    nan = np.isnan(x)
    out = r.astype(np.uint32).view(np.float32).copy()
    out[nan] = np.nan
    return out
