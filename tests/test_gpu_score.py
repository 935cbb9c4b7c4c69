"""GPU parity of the local score (through the C ABI) against the fp64 oracle:
delta[k][s] = <g_s, delta_o[k][s]>, the loss change whose reduction is the
Dust page's c_s = -<g_s, delta_o_s> ("What the released code actually does",
step 4).

Tolerance: fp32 products of exact bf16/fp32 inputs summed in fp32 over d
terms, 1e-5 normwise relative for d <= 1024 (the per-row relative error of a
d-term fp32 sum is about sqrt(d) 2^-24 for random signs).
"""
import numpy as np
import pytest

import oracle
import token_perturbation_estimator_gb300 as dust
from helpers import cuda, offsets_from_lengths, random_lengths, rel_fro

pytestmark = pytest.mark.gpu

CASES = [
    # K, T, d, g dtype, delta_o dtype
    (1, 1, 1, "f32", "f32"),
    (3, 37, 33, "f32", "bf16"),     # d not a multiple of 8: scalar loads
    (8, 1000, 512, "bf16", "bf16"),  # 16-byte vector loads
    (4, 300, 136, "bf16", "f32"),
    (2, 64, 1024, "f32", "f32"),
    (16, 129, 8, "bf16", "bf16"),   # one vector per lane-row
]


def _tensor(x, dtype, dev):
    import torch
    t = torch.from_numpy(x.astype(np.float32)).to(dev)
    return t.to(torch.bfloat16) if dtype == "bf16" else t


@pytest.mark.parametrize("K,T,d,gd,od", CASES)
def test_local_score_parity(K, T, d, gd, od):
    dev = cuda()
    rng = np.random.default_rng(K * 100 + d)
    g = _tensor(rng.standard_normal((T, d)), gd, dev)
    dO = _tensor(rng.standard_normal((K, T, d)), od, dev)
    got = dust.dust_local_score(g, dO).double().cpu().numpy()
    want = oracle.local_score(g.double().cpu().numpy(), dO.double().cpu().numpy())
    assert rel_fro(got, want) <= 1e-5
    again = dust.dust_local_score(g, dO).double().cpu().numpy()
    assert np.array_equal(got, again)


def test_empty_and_zero_width():
    import torch
    dev = cuda()
    out = torch.full((2, 3), 7.0, device=dev)
    dust.dust_local_score(torch.empty((3, 0), device=dev), torch.empty((2, 3, 0), device=dev),
                          out=out)
    assert torch.count_nonzero(out).item() == 0
    dust.dust_local_score(torch.empty((0, 4), device=dev), torch.empty((2, 0, 4), device=dev))


@pytest.mark.slow
def test_attention_block_scores_drive_the_estimate():
    """A value projection (512 -> 512) of an attention block at the measured
    size (16 x 1024 tokens, K = 8): scores from the block output's error and
    its changes under the draws feed the estimator with gamma 0.98 over later
    tokens; the estimate matches the oracle run on the same inputs."""
    import torch
    dev = cuda()
    rng = np.random.default_rng(7)
    T, d, K, d_in = 16384, 512, 8, 512
    so = offsets_from_lengths([1024] * 16)
    g = _tensor(rng.standard_normal((T, d)), "bf16", dev)
    dO = _tensor(1e-3 * rng.standard_normal((K, T, d)), "bf16", dev)
    delta = dust.dust_local_score(g, dO)
    want_delta = oracle.local_score(g.double().cpu().numpy(), dO.double().cpu().numpy())
    assert rel_fro(delta.double().cpu().numpy(), want_delta) <= 1e-5
    X = _tensor(rng.standard_normal((T, d_in)), "bf16", dev)
    got = dust.dust_estimate_gW(X, delta, d, torch.from_numpy(so).to(dev), 3, dust.GAUSSIAN, 0,
                                1e-3, 0.98, 1.0 / T, dust.CENTER).double().cpu().numpy()
    # entries of the oracle's estimate from the GPU's scores, one by one
    r = oracle.credit(delta.double().cpu().numpy(), so, np.float32(0.98), oracle.CENTER)
    chan = rng.integers(0, d, 32)
    col = rng.integers(0, d_in, 32)
    want = oracle.gW_entries(X.double().cpu().numpy(), r, d, chan, col, 3, dust.GAUSSIAN, 0,
                             np.float32(1e-3), 1.0 / T, oracle.CENTER)
    assert rel_fro(got[chan, col], want) <= 1e-2
