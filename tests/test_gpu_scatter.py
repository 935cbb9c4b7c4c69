"""GPU parity of the embedding reassembly (dust_scatter_gE) and the whole
embedding estimator (dust_estimate_gE) against the fp64 oracle ("Dust: every
token is a member of the population", "What the released code actually
does", step 7: a scatter-add for an embedding).

Tolerances: the scatter keeps 64-bit fixed-point sums (each term rounded to a
step far below its magnitude) and rounds once to fp32, so 1e-6 normwise
relative; the estimator adds the weighting's fp32 arithmetic, 1e-5.
"""
import numpy as np
import pytest

import oracle
import token_perturbation_estimator_gb300 as dust
from helpers import cuda, offsets_from_lengths, random_lengths, rel_fro

pytestmark = pytest.mark.gpu


def _zipf_ids(rng, T, V):
    """Token ids with the heavy repetition of natural text (Zipf, s = 1.1)."""
    ranks = rng.zipf(1.1, T * 2)
    ranks = ranks[ranks <= V][:T]
    while ranks.size < T:
        ranks = np.concatenate([ranks, rng.integers(1, V + 1, T - ranks.size)])
    return (ranks - 1).astype(np.int32)


CASES = [
    # T, d, V, ids, g dtype
    (1000, 33, 100, "uniform", "f32"),
    (20000, 512, 4096, "zipf", "bf16"),
    (777, 64, 5, "uniform", "f32"),   # few ids: long sums per row
    (1, 8, 1, "uniform", "f32"),
]


@pytest.mark.parametrize("T,d,V,dist,gd", CASES)
def test_scatter_parity_and_determinism(T, d, V, dist, gd):
    import torch
    dev = cuda()
    rng = np.random.default_rng(T + d)
    ids = _zipf_ids(rng, T, V) if dist == "zipf" else rng.integers(0, V, T).astype(np.int32)
    g = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(dev)
    if gd == "bf16":
        g = g.to(torch.bfloat16)
    idd = torch.from_numpy(ids).to(dev)
    got = dust.dust_scatter_gE(g, idd, V, 0.5)
    want, bad = oracle.scatter_gE(g.double().cpu().numpy(), ids, V, 0.5)
    assert bad == 0
    assert rel_fro(got.double().cpu().numpy(), want) <= 1e-6
    again = dust.dust_scatter_gE(g, idd, V, 0.5)
    assert torch.equal(got, again)
    base = torch.randn((V, d), device=dev)
    acc = dust.dust_scatter_gE(g, idd, V, 0.5, flags=dust.ACCUMULATE, gE=base.clone())
    assert torch.allclose(acc, base + got, rtol=1e-6, atol=1e-6 * got.abs().max().item())
    assert dust.dust_last_error() == dust.OK


def test_one_id_and_zero_rows():
    import torch
    dev = cuda()
    T, d, V = 4096, 40, 10
    g = torch.randn((T, d), device=dev)
    ids = torch.full((T,), 7, dtype=torch.int32, device=dev)
    got = dust.dust_scatter_gE(g, ids, V).cpu()
    assert torch.count_nonzero(got[:7]).item() == 0 and torch.count_nonzero(got[8:]).item() == 0
    want = g.double().sum(dim=0).cpu()
    assert torch.allclose(got[7].double(), want, rtol=1e-6, atol=1e-5)
    zero = dust.dust_scatter_gE(torch.zeros((T, d), device=dev), ids, V)
    assert torch.count_nonzero(zero).item() == 0


def test_out_of_range_ids_are_skipped_and_reported():
    import torch
    dev = cuda()
    g = torch.ones((6, 4), device=dev)
    ids = torch.tensor([0, 9, 2, -1, 2, 3], dtype=torch.int32, device=dev)
    got = dust.dust_scatter_gE(g, ids, 4).cpu()
    assert dust.dust_last_error() == dust.ERR_INVALID_ARG
    assert dust.dust_last_error() == dust.OK  # cleared
    want = torch.tensor([[1.0] * 4, [0.0] * 4, [2.0] * 4, [1.0] * 4])
    assert torch.equal(got, want)


@pytest.mark.parametrize("kind,flags", [(dust.GAUSSIAN, dust.CENTER),
                                        (dust.RADEMACHER_PACKED, dust.CENTER | dust.ANTITHETIC)])
def test_embedding_estimate_matches_oracle(kind, flags):
    import torch
    dev = cuda()
    rng = np.random.default_rng(17)
    T, d, V, K = 3000, 96, 500, 8
    so = offsets_from_lengths(random_lengths(rng, T, 700))
    ids = _zipf_ids(rng, T, V)
    delta = (0.05 * rng.standard_normal((K, T))).astype(np.float32)
    got = dust.dust_estimate_gE(torch.from_numpy(ids).to(dev), torch.from_numpy(delta).to(dev),
                                V, d, torch.from_numpy(so).to(dev), 5, kind, 2, 1e-3, 0.9,
                                1.0 / T, flags).double().cpu().numpy()
    oflags = flags & (oracle.CENTER | oracle.ANTITHETIC)
    r = oracle.credit(delta, so, np.float32(0.9), oflags)
    g = oracle.error_estimate(r, d, 5, kind, 2, np.float32(1e-3), oflags)
    want, _ = oracle.scatter_gE(g, ids, V, 1.0 / T)
    assert rel_fro(got, want) <= 1e-5
