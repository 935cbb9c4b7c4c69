"""GPU parity of the jittered forward (dust_forward_jitter) against the fp64
oracle ("Dust: every token is a member of the population", section "Perturb
the activations, not the weights": each draw's output is the layer's product
plus sigma times that draw's jitter).

Error bound, per element. The kernel accumulates y = X W^T in fp32 on the
tensor cores from exact bf16 products, adds sigma a in fp32 and rounds once to
bf16 (nearest even). With z the fp32 value before the rounding and w the fp64
oracle value:
    |z - w| <= e = d_in 2^-22 sum_j |x_j w_j| + sigma 1e-5 max(1, |a|)
(fp32 accumulation over d_in terms; the Gaussian jitter's fp32 evaluation is
within 1e-5 max(1, |a|) of the fp64 one, Rademacher signs are exact), and
the bf16 rounding adds at most 2^-8 |z| <= 2^-8 (|w| + e).
"""
import time

import numpy as np
import pytest

import oracle
import token_perturbation_estimator_gb300 as dust
from helpers import bf16_round, cuda

pytestmark = pytest.mark.gpu


def _inputs(T, d_in, d_out, seed, w_zero=False):
    rng = np.random.default_rng(seed)
    X = bf16_round(rng.standard_normal((T, d_in)))
    W = np.zeros((d_out, d_in)) if w_zero else bf16_round(
        rng.standard_normal((d_out, d_in)) / np.sqrt(d_in))
    return X, W


def _to_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).to(dev)


def _bound(X, W, want, sigma, noise_abs):
    d_in = X.shape[1]
    s_abs = np.abs(X) @ np.abs(W).T  # [T, d_out]
    e = d_in * 2.0 ** -22 * s_abs[None] + sigma * 1e-5 * np.maximum(1.0, noise_abs)
    return 2.0 ** -8 * (np.abs(want) + e) + e


SHAPES = [
    # T, d_in, d_out
    (128, 64, 256),     # one tile, one k-step
    (300, 72, 200),     # ragged tokens, d_in (zero-filled k-step) and channels
    (1000, 520, 520),   # three channel tiles, ragged
    (64, 8, 8),         # smallest legal layer
    (2048, 1024, 768),  # 16 token tiles x 3 channel tiles, 16 k-steps
]


@pytest.mark.parametrize("T,d_in,d_out", SHAPES)
@pytest.mark.parametrize("kind", [dust.RADEMACHER, dust.GAUSSIAN, dust.RADEMACHER_PACKED])
def test_forward_matches_oracle(T, d_in, d_out, kind):
    dev = cuda()
    X, W = _inputs(T, d_in, d_out, T + d_in + kind)
    sigma, n_draws, draw_begin = 0.25, 3, 5
    got = dust.dust_forward_jitter(_to_dev(X, dev), _to_dev(W, dev), 11, kind, draw_begin,
                                   n_draws, sigma, clean=True)
    assert dust.dust_last_error() == dust.OK
    want = oracle.forward_jitter(X, W, 11, kind, draw_begin, n_draws, sigma, clean=True)
    a = np.abs(want[1:] - want[:1]) / sigma
    bound = _bound(X, W, want, sigma, np.concatenate([np.zeros((1,) + a.shape[1:]), a]))
    err = np.abs(got.double().cpu().numpy() - want)
    assert (err <= bound).all(), float((err - bound).max())


@pytest.mark.parametrize("kind", [dust.RADEMACHER, dust.RADEMACHER_PACKED])
@pytest.mark.parametrize("flags,draw_begin", [(0, 0), (dust.ANTITHETIC, 3)])
def test_signs_bit_exact_when_the_product_is_zero(kind, flags, draw_begin):
    """W = 0: every slice is bf16(sigma a) = +-sigma exactly (sigma = 0.5)."""
    import torch
    dev = cuda()
    T, d_in, d_out = 300, 64, 200
    X, W = _inputs(T, d_in, d_out, 1, w_zero=True)
    got = dust.dust_forward_jitter(_to_dev(X, dev), _to_dev(W, dev), 99, kind, draw_begin, 5,
                                   0.5, flags=flags, clean=True)
    want = oracle.forward_jitter(X, W, 99, kind, draw_begin, 5, 0.5, flags=flags, clean=True)
    assert torch.count_nonzero(got[0]).item() == 0
    assert np.array_equal(got.double().cpu().numpy(), want)


@pytest.mark.parametrize("flags", [0, dust.ANTITHETIC])
def test_gaussian_jitter_alone(flags):
    """W = 0: the slices are the rounded Gaussian jitter sigma a."""
    dev = cuda()
    T, d_in, d_out = 256, 64, 512
    X, W = _inputs(T, d_in, d_out, 2, w_zero=True)
    got = dust.dust_forward_jitter(_to_dev(X, dev), _to_dev(W, dev), 5, dust.GAUSSIAN, 1, 4,
                                   2.0, flags=flags).double().cpu().numpy()
    want = oracle.forward_jitter(X, W, 5, oracle.GAUSSIAN, 1, 4, 2.0, flags=flags)
    e = 2.0 * 1e-5 * np.maximum(1.0, np.abs(want) / 2.0)
    assert (np.abs(got - want) <= 2.0 ** -8 * (np.abs(want) + e) + e).all()


def test_many_draws_and_no_clean_slice():
    """More draws than the kernel's shared key table (64): the rest are keyed inline."""
    dev = cuda()
    T, d_in, d_out = 256, 64, 64
    X, W = _inputs(T, d_in, d_out, 3)
    got = dust.dust_forward_jitter(_to_dev(X, dev), _to_dev(W, dev), 8, dust.GAUSSIAN, 100, 70,
                                   0.5, flags=dust.ANTITHETIC)
    want = oracle.forward_jitter(X, W, 8, oracle.GAUSSIAN, 100, 70, 0.5, flags=oracle.ANTITHETIC)
    a = np.abs(want - (X @ W.T)[None]) / 0.5
    err = np.abs(got.double().cpu().numpy() - want)
    assert (err <= _bound(X, W, want, 0.5, a)).all()


def test_clean_slice_only_and_determinism():
    import torch
    dev = cuda()
    T, d_in, d_out = 1000, 512, 1024
    X, W = _inputs(T, d_in, d_out, 4)
    Xd, Wd = _to_dev(X, dev), _to_dev(W, dev)
    got = dust.dust_forward_jitter(Xd, Wd, 0, dust.GAUSSIAN, 0, 0, 1.0, clean=True)
    want = X @ W.T
    err = np.abs(got[0].double().cpu().numpy() - want)
    assert (err <= _bound(X, W, want[None], 0.0, np.zeros((1,) + want.shape))[0]).all()
    again = dust.dust_forward_jitter(Xd, Wd, 0, dust.GAUSSIAN, 0, 0, 1.0, clean=True)
    assert torch.equal(got, again)
    # sigma = 0: every draw slice repeats the clean one bit for bit
    rep = dust.dust_forward_jitter(Xd, Wd, 0, dust.GAUSSIAN, 0, 3, 0.0, clean=True)
    for s in range(4):
        assert torch.equal(rep[s], got[0])


def test_full_size_mlp_up_sampled():
    """The measured layer (16384 tokens, 512 -> 2048, 8 Gaussian draws plus the
    clean slice, sigma 1e-3), checked on sampled outputs element by element."""
    import torch
    dev = cuda()
    T, d_in, d_out, K, sigma = 16384, 512, 2048, 8, 1e-3
    gen = torch.Generator().manual_seed(6)
    Xd = torch.randn((T, d_in), generator=gen).to(torch.bfloat16).to(dev)
    Wd = (torch.randn((d_out, d_in), generator=gen) / np.sqrt(d_in)).to(torch.bfloat16).to(dev)
    Y = dust.dust_forward_jitter(Xd, Wd, 0, dust.GAUSSIAN, 0, K, sigma, clean=True)
    assert dust.dust_last_error() == dust.OK
    rng = np.random.default_rng(7)
    n = 4000
    s = rng.integers(0, K + 1, n)
    t = rng.integers(0, T, n)
    c = rng.integers(0, d_out, n)
    Xs = Xd.double().cpu().numpy()[t]
    Ws = Wd.double().cpu().numpy()[c]
    y = (Xs * Ws).sum(axis=1)
    a = np.zeros(n)
    m = s > 0
    a[m] = oracle.noise_at(s[m] - 1, t[m], c[m], 0, oracle.GAUSSIAN, d_out)
    want = y + sigma * a
    got = Y[torch.from_numpy(s).to(dev), torch.from_numpy(t).to(dev),
            torch.from_numpy(c).to(dev)].double().cpu().numpy()
    e = d_in * 2.0 ** -22 * (np.abs(Xs) * np.abs(Ws)).sum(axis=1) + sigma * 1e-5 * np.maximum(1, np.abs(a))
    assert (np.abs(got - want) <= 2.0 ** -8 * (np.abs(want) + e) + e).all()


def test_bounded_wait_timeout_is_reported_and_context_survives():
    import torch
    dev = cuda()
    T, d_in, d_out = 512, 256, 512
    X, W = _inputs(T, d_in, d_out, 9)
    Xd, Wd = _to_dev(X, dev), _to_dev(W, dev)
    assert dust.dust_last_error() == dust.OK
    dust.lib().dust_debug_inject_timeout(1)
    t0 = time.time()
    dust.dust_forward_jitter(Xd, Wd, 1, dust.RADEMACHER, 0, 2, 0.5, clean=True)
    st = dust.dust_last_error()
    assert st == dust.ERR_TIMEOUT, dust.status_string(st)
    assert 0.5 < time.time() - t0 < 30.0
    assert dust.dust_last_error() == dust.OK
    got = dust.dust_forward_jitter(Xd, Wd, 1, dust.RADEMACHER, 0, 2, 0.5, clean=True)
    want = oracle.forward_jitter(X, W, 1, oracle.RADEMACHER, 0, 2, 0.5, clean=True)
    a = np.concatenate([np.zeros((1, T, d_out)), np.ones((2, T, d_out))])
    assert (np.abs(got.double().cpu().numpy() - want) <= _bound(X, W, want, 0.5, a)).all()
    assert dust.dust_last_error() == dust.OK


@pytest.mark.parametrize("kind", [dust.RADEMACHER, dust.GAUSSIAN, dust.RADEMACHER_PACKED])
def test_largest_counter_range_sampled(kind):
    """T d_out = 2^32 (the counter's whole range, 65536 tokens x 65536 channels,
    131072 tiles, one 8.6 GB slice): sampled outputs, including the last
    token's last channels, against the oracle element by element."""
    import torch
    dev = cuda()
    T, d_in, d_out, sigma = 65536, 8, 65536, 0.5
    gen = torch.Generator().manual_seed(11)
    Xd = torch.randn((T, d_in), generator=gen).to(torch.bfloat16).to(dev)
    Wd = torch.randn((d_out, d_in), generator=gen).to(torch.bfloat16).to(dev)
    Y = dust.dust_forward_jitter(Xd, Wd, 77, kind, 1000, 1, sigma)
    assert dust.dust_last_error() == dust.OK
    rng = np.random.default_rng(12)
    n = 3000
    t = np.concatenate([rng.integers(0, T, n), np.full(64, T - 1)])
    c = np.concatenate([rng.integers(0, d_out, n), np.arange(d_out - 64, d_out)])
    Xs = Xd[torch.from_numpy(t).to(dev)].double().cpu().numpy()
    Ws = Wd[torch.from_numpy(c).to(dev)].double().cpu().numpy()
    a = oracle.noise_at(np.full(t.size, 1000), t, c, 77, kind, d_out)
    want = (Xs * Ws).sum(axis=1) + sigma * a
    got = Y[0, torch.from_numpy(t).to(dev), torch.from_numpy(c).to(dev)].double().cpu().numpy()
    e = d_in * 2.0 ** -22 * (np.abs(Xs) * np.abs(Ws)).sum(axis=1) + sigma * 1e-5 * np.maximum(1, np.abs(a))
    assert (np.abs(got - want) <= 2.0 ** -8 * (np.abs(want) + e) + e).all()
    del Y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind,flags", [(dust.GAUSSIAN, 0), (dust.RADEMACHER_PACKED, dust.ANTITHETIC)])
def test_highest_draw_indices(kind, flags):
    """The last legal draws (draw_begin + n_draws = 2^31): keys made from the
    largest absolute indices, more of them than the shared key table holds."""
    dev = cuda()
    T, d_in, d_out = 200, 64, 96
    X, W = _inputs(T, d_in, d_out, 13)
    n = 66
    db = (1 << 31) - n
    got = dust.dust_forward_jitter(_to_dev(X, dev), _to_dev(W, dev), 2 ** 40 + 7, kind, db, n,
                                   0.5, flags=flags)
    assert dust.dust_last_error() == dust.OK
    want = oracle.forward_jitter(X, W, 2 ** 40 + 7, kind, db, n, 0.5, flags=flags)
    a = np.abs(want - (X @ W.T)[None]) / 0.5
    err = np.abs(got.double().cpu().numpy() - want)
    assert (err <= _bound(X, W, want, 0.5, a)).all()
