"""Pins for the oracle's noise values (CPU only).

What the pages fix: the jitter a_t ~ N(0, I) of "Dust: every token is a
member of the population" ("Perturb the activations, not the weights"), with
E[a a^T] = I ("What a zeroth-order gradient is"); Rademacher signs are
zero-mean, unit-variance and symmetric ("RandOpt Speedrun", "What was slow,
and the fix"). The Gaussian is checked against the normal CDF (scipy), not
against a retyped Box-Muller.
"""
import numpy as np
import pytest
from scipy import stats


def test_rademacher_exact_signs_and_balance(orc):
    a = orc.noise(seed=11, kind=orc.RADEMACHER, draw_begin=0, n_draws=4, T=2048, d_out=1024)
    assert set(np.unique(a).tolist()) == {-1.0, 1.0}
    n = a.size
    assert abs(a.mean()) <= 4.0 / np.sqrt(n)
    # adjacent channel, adjacent token and cross-draw correlations
    for x, y in ((a[..., 1:], a[..., :-1]), (a[:, 1:, :], a[:, :-1, :]), (a[1:], a[:-1])):
        m = x.size
        assert abs(np.mean(x * y)) <= 4.0 / np.sqrt(m)


def test_rademacher_sign_is_top_bit_of_stream0_word(orc):
    w = orc.words(seed=5, draw_begin=2, n_draws=3, T=64, d_out=33, stream=0)
    a = orc.noise(seed=5, kind=orc.RADEMACHER, draw_begin=2, n_draws=3, T=64, d_out=33)
    assert np.array_equal(a, np.where(w >> 31, -1.0, 1.0))


@pytest.mark.parametrize("kind", [0, 1])
def test_second_moment_is_identity(orc, kind):
    """E[a a^T] = I over a d-dimensional token jitter."""
    d = 16
    a = orc.noise(seed=3, kind=kind, draw_begin=0, n_draws=8, T=20000, d_out=d).reshape(-1, d)
    n = a.shape[0]
    C = a.T @ a / n
    assert np.max(np.abs(C - np.eye(d))) <= 5.0 * np.sqrt(3.0 / n)


def test_gaussian_marginal_is_standard_normal(orc):
    a = orc.noise(seed=21, kind=orc.GAUSSIAN, draw_begin=0, n_draws=2, T=4096, d_out=130)
    x = a.ravel()
    n = x.size
    assert abs(x.mean()) <= 5.0 / np.sqrt(n)
    assert abs(x.var() - 1.0) <= 5.0 * np.sqrt(2.0 / n)
    assert abs(np.mean(x ** 4) - 3.0) <= 5.0 * np.sqrt(96.0 / n)
    # both halves of each Box-Muller pair, separately
    for half in (x.reshape(-1, 2)[:, 0], x.reshape(-1, 2)[:, 1]):
        assert stats.kstest(half, "norm").pvalue > 1e-4
    ev, od = a[..., 0::2].ravel(), a[..., 1::2].ravel()
    assert abs(np.mean(ev * od)) <= 5.0 / np.sqrt(ev.size)
    # the radius rho^2 = a_p^2 + a_{p+1}^2 is chi-square with 2 dof
    rho2 = ev ** 2 + od ** 2
    assert stats.kstest(rho2, "chi2", args=(2,)).pvalue > 1e-4


def test_gaussian_odd_width_last_channel_is_cos_branch(orc):
    """With odd d_out the last channel has no sine partner; its value is the
    cosine half of its own pair, so it is still N(0, 1)."""
    a = orc.noise(seed=4, kind=orc.GAUSSIAN, draw_begin=0, n_draws=1, T=40000, d_out=5)
    last = a[0, :, 4]
    assert stats.kstest(last, "norm").pvalue > 1e-4


def test_antithetic_pairs_are_exact_negatives(orc):
    f = orc.ANTITHETIC
    for kind in (0, 1):
        a = orc.noise(seed=9, kind=kind, draw_begin=0, n_draws=6, T=32, d_out=17, flags=f)
        assert np.array_equal(a[1::2], -a[0::2])
        base = orc.noise(seed=9, kind=kind, draw_begin=0, n_draws=3, T=32, d_out=17)
        assert np.array_equal(a[0::2], base)


def test_draw_split_reproducible(orc):
    for kind in (0, 1):
        full = orc.noise(seed=77, kind=kind, draw_begin=0, n_draws=7, T=20, d_out=9)
        part = orc.noise(seed=77, kind=kind, draw_begin=3, n_draws=3, T=20, d_out=9)
        assert np.array_equal(full[3:6], part)
        again = orc.noise(seed=77, kind=kind, draw_begin=0, n_draws=7, T=20, d_out=9)
        assert np.array_equal(full, again)


def test_noise_at_matches_dense(orc):
    full = orc.noise(seed=1, kind=1, draw_begin=0, n_draws=3, T=10, d_out=7)
    rng = np.random.default_rng(0)
    i = rng.integers(0, 3, 50)
    t = rng.integers(0, 10, 50)
    c = rng.integers(0, 7, 50)
    assert np.array_equal(orc.noise_at(i, t, c, 1, 1, 7), full[i, t, c])


def test_different_seeds_are_uncorrelated(orc):
    a = orc.noise(seed=100, kind=1, draw_begin=0, n_draws=1, T=1000, d_out=200).ravel()
    b = orc.noise(seed=101, kind=1, draw_begin=0, n_draws=1, T=1000, d_out=200).ravel()
    assert abs(np.mean(a * b)) <= 5.0 / np.sqrt(a.size)


# ------------------------------------------------- packed Rademacher signs --
# Thirty-two signs per hash word (a noise kind of this project, motivated by
# "RandOpt Speedrun", "What was slow, and the fix": the hash is the cost, so
# spend every bit of it): channel c takes bit c mod 32 of the stream-0 word at
# the counter of its group's first channel 32 floor(c / 32); bit 0 gives +1.

def test_packed_sign_is_bit_of_group_word(orc):
    T, d_out = 40, 77  # three groups, the last one 13 channels wide
    w = orc.words(seed=6, draw_begin=1, n_draws=3, T=T, d_out=d_out, stream=0)
    a = orc.noise(seed=6, kind=orc.RADEMACHER_PACKED, draw_begin=1, n_draws=3, T=T,
                  d_out=d_out)
    c = np.arange(d_out)
    word = w[..., (c // 32) * 32]
    bit = (word >> (c % 32).astype(np.uint32)) & np.uint32(1)
    assert np.array_equal(a, np.where(bit == 1, -1.0, 1.0))


def test_packed_top_bit_channel_equals_per_channel_sign(orc):
    """Channel 32q + 31 reads the top bit of the word at counter 32q, which is
    exactly the per-channel Rademacher sign of channel 32q."""
    a = orc.noise(seed=8, kind=orc.RADEMACHER_PACKED, draw_begin=0, n_draws=2, T=50,
                  d_out=96)
    r = orc.noise(seed=8, kind=orc.RADEMACHER, draw_begin=0, n_draws=2, T=50, d_out=96)
    for q in range(3):
        assert np.array_equal(a[..., 32 * q + 31], r[..., 32 * q])


def test_packed_signs_balance_and_independence(orc):
    a = orc.noise(seed=12, kind=orc.RADEMACHER_PACKED, draw_begin=0, n_draws=4, T=2048,
                  d_out=1024)
    assert set(np.unique(a).tolist()) == {-1.0, 1.0}
    assert abs(a.mean()) <= 4.0 / np.sqrt(a.size)
    # neighbouring bits of one word, the same bit of neighbouring words,
    # neighbouring tokens and draws
    pairs = ((a[..., 1:], a[..., :-1]), (a[..., 32:], a[..., :-32]),
             (a[:, 1:, :], a[:, :-1, :]), (a[1:], a[:-1]))
    for x, y in pairs:
        assert abs(np.mean(x * y)) <= 4.0 / np.sqrt(x.size)
    # every bit position is balanced on its own
    for b in range(32):
        col = a[..., b::32]
        assert abs(col.mean()) <= 5.0 / np.sqrt(col.size)


def test_packed_antithetic_and_draw_split(orc):
    f = orc.ANTITHETIC
    k = orc.RADEMACHER_PACKED
    a = orc.noise(seed=9, kind=k, draw_begin=0, n_draws=6, T=32, d_out=70, flags=f)
    assert np.array_equal(a[1::2], -a[0::2])
    full = orc.noise(seed=77, kind=k, draw_begin=0, n_draws=7, T=20, d_out=40)
    part = orc.noise(seed=77, kind=k, draw_begin=3, n_draws=3, T=20, d_out=40)
    assert np.array_equal(full[3:6], part)
