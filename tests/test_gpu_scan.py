"""GPU parity of centring + the segmented reverse credit scan (through the C
ABI) against the fp64 oracle: normwise relative error <= 1e-5 on r [T, K],
over ragged sequence sets, chunk-crossing sequences and edge cases."""
import numpy as np
import pytest

import oracle
import token_perturbation_estimator_gb300 as dust
from helpers import cuda, offsets_from_lengths, random_lengths, rel_fro

pytestmark = pytest.mark.gpu

CASES = [
    # K, T, max sequence length, gamma, centre
    (1, 1, 1, 0.9, True),
    (2, 255, 40, 0.0, True),
    (4, 256, 256, 0.9, True),
    (7, 257, 300, 0.5, False),
    (8, 16384, 1024, 0.0, True),
    (16, 5000, 2048, 0.9, True),
    (33, 3000, 1, 0.9, True),        # one-token sequences only
    (64, 2048, 2048, 1.0, True),     # undiscounted reward-to-go
    (100, 1000, 37, 0.98, True),
    (3, 20000, 20000, 0.999, False),  # one long sequence across many chunks
    (5, 65536, 65536, 0.999, False),  # one sequence over 256 chunks
    (2, 40000, 2, 0.9, True),         # > 4096 sequences: per-token offset search
    (256, 600, 100, 0.9, True),       # many draws: several draw groups per chunk
    (257, 600, 100, 0.9, True),       # a one-draw last group
    (4, 70000, 5000, 0.99, True),
    (2, 65537, 65537, 1.0, False),    # one undiscounted sequence, a 1-token last chunk
    (8, 300000, 300000, 0.9999, False),  # too many chunk summaries to merge: separate carry kernel
    (4, 300000, 300000, 0.99999, False),  # a horizon of about 390 chunks
    (4, 300000, 300000, -0.9999, False),  # alternating decay
    (4, 300000, 300000, 1.0, True),       # undiscounted, centred, 1172 chunks
    (32, 65536, 1024, 0.9, True),         # the sweep's QKV sites
]


@pytest.mark.parametrize("K,T,max_len,gamma,center", CASES)
def test_credit_scan_parity(K, T, max_len, gamma, center):
    import torch
    dev = cuda()
    rng = np.random.default_rng(K * 1000 + T)
    lengths = random_lengths(rng, T, max_len)
    so = offsets_from_lengths(lengths)
    delta = (0.05 * rng.standard_normal((K, T)) + 0.01).astype(np.float32)
    flags = dust.CENTER if center else 0
    r = dust.dust_credit_scan(torch.from_numpy(delta).to(dev), torch.from_numpy(so).to(dev),
                              gamma, flags)
    got = r.cpu().numpy().T  # [K, T]
    want = oracle.credit(delta, so, np.float32(gamma), flags)
    assert got.shape == want.shape
    assert rel_fro(got, want) <= 1e-5
    assert np.max(np.abs(got - want)) <= 1e-5 * np.abs(want).max()


def test_credit_scan_gamma_zero_is_centred_reduction():
    import torch
    dev = cuda()
    rng = np.random.default_rng(5)
    K, T = 6, 700
    delta = rng.standard_normal((K, T)).astype(np.float32)
    so = offsets_from_lengths([300, 400])
    r = dust.dust_credit_scan(torch.from_numpy(delta).to(dev), torch.from_numpy(so).to(dev),
                              0.0, dust.CENTER).cpu().numpy().T
    c = -(delta.astype(np.float64) - delta.astype(np.float64).mean(axis=0))
    assert np.max(np.abs(r - c)) <= 1e-6
    assert np.max(np.abs(r.sum(axis=0))) <= 1e-5

