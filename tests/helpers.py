"""Shared helpers for the GPU parity tests."""
import numpy as np
import pytest


def cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a visible CUDA device")
    import token_perturbation_estimator_gb300 as dust
    from token_perturbation_estimator_gb300 import build
    build.build()
    dust.lib()
    return torch.device("cuda:0")


def rel_fro(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def offsets_from_lengths(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def random_lengths(rng, T, max_len):
    out, left = [], T
    while left > 0:
        n = int(min(left, rng.integers(1, max_len + 1)))
        out.append(n)
        left -= n
    return out


def bf16_round(x):
    """Round float64 values to bf16 (through float32, nearest-even)."""
    import workloads
    return workloads.to_bf16_exact(np.asarray(x, np.float32)).astype(np.float64)
