"""Pins for the oracle's estimator steps (CPU only).

The three equations of "Dust: every token is a member of the population",
section "Perturb the activations, not the weights":
    r_t = sum_{s>=t} gamma^(s-t) c_s,  g_t = -(1/(K sigma)) sum_i r_t^(i) a_t^(i),
    GW = sum_t g_t x_t^T,
with c the centred loss reduction ("What the released code actually does",
step 2). Pins: closed forms of the scan, the centring invariant, the
unbiasedness of the estimate under a planted linear loss (E[a a^T] = I,
"What a zeroth-order gradient is"), the antithetic cancellation of even-order
terms (same section), the cosine law sqrt(K/(K+D)) and the page's toy
cosines (tests/golden), and a brute-force triple sum on tiny inputs.
"""
import os

import numpy as np
import pytest

GOLDEN_TOY = os.path.join(os.path.dirname(__file__), "golden", "toy_per_token_cosine.txt")


def _offsets(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


# ---------------------------------------------------------------- centring --

def test_center_sums_to_zero_and_negates(orc):
    rng = np.random.default_rng(0)
    d = rng.standard_normal((6, 50))
    c = orc.center(d, orc.CENTER)
    assert np.allclose(c.sum(axis=0), 0.0, atol=1e-13)
    assert np.allclose(c, -(d - d.mean(axis=0)), atol=1e-14)
    assert np.array_equal(orc.center(d, 0), -d)


def test_center_single_draw_is_noop(orc):
    d = np.random.default_rng(1).standard_normal((1, 40))
    assert np.array_equal(orc.center(d, orc.CENTER), -d)


# -------------------------------------------------------------------- scan --

def test_scan_gamma_zero_is_identity(orc):
    c = np.random.default_rng(2).standard_normal((3, 100))
    assert np.array_equal(orc.scan(c, _offsets([30, 1, 69]), 0.0), c)


@pytest.mark.parametrize("gamma", [0.3, 0.9, 0.98, 1.0])
def test_scan_constant_closed_form(orc, gamma):
    """For constant c the reward-to-go at distance k from the sequence end is
    c (1 - gamma^(k+1)) / (1 - gamma) (c (k+1) at gamma = 1)."""
    lengths = [17, 1, 40]
    T = sum(lengths)
    c = np.full((2, T), 0.75)
    r = orc.scan(c, _offsets(lengths), gamma)
    o = _offsets(lengths)
    for q in range(len(lengths)):
        for t in range(o[q], o[q + 1]):
            k = o[q + 1] - 1 - t
            want = 0.75 * (k + 1) if gamma == 1.0 else 0.75 * (1 - gamma ** (k + 1)) / (1 - gamma)
            assert r[0, t] == pytest.approx(want, rel=1e-12)


def test_scan_matches_discounted_sum_definition(orc):
    """The recurrence equals the sum definition r_t = sum_{s>=t, same sequence}
    gamma^(s-t) c_s, evaluated here as an explicit discount matrix."""
    rng = np.random.default_rng(3)
    lengths = [5, 1, 12, 7]
    o = _offsets(lengths)
    T = int(o[-1])
    c = rng.standard_normal((4, T))
    gamma = 0.8
    D = np.zeros((T, T))
    for q in range(len(lengths)):
        for t in range(o[q], o[q + 1]):
            for s in range(t, o[q + 1]):
                D[t, s] = gamma ** (s - t)
    assert np.allclose(orc.scan(c, o, gamma), c @ D.T, rtol=1e-13, atol=1e-13)


def test_scan_one_token_sequences(orc):
    c = np.random.default_rng(4).standard_normal((2, 9))
    assert np.array_equal(orc.scan(c, np.arange(10, dtype=np.int32), 0.9), c)


# ------------------------------------------------------- brute-force sums --

@pytest.mark.parametrize("kind", [0, 1, 3])
@pytest.mark.parametrize("flags", [0, 1, 3])
def test_pipeline_equals_brute_force(orc, kind, flags):
    rng = np.random.default_rng(5)
    lengths = [7, 1, 9]
    o = _offsets(lengths)
    T, d_in, d_out, K = int(o[-1]), 5, 6, 4
    X = rng.standard_normal((T, d_in))
    delta = rng.standard_normal((K, T))
    args = dict(seed=42, kind=kind, draw_begin=3, sigma=0.01, gamma=0.7, scale=0.5, flags=flags)
    a = orc.estimate_gW(X, delta, d_out, o, **args)
    b = orc.bruteforce_gW(X, delta, d_out, o, **args)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12 * np.abs(b).max())


def test_weighting_and_contraction_definitions(orc):
    """g from the scan output and the oracle's own noise, contracted with X,
    equals einsum of the definitions."""
    rng = np.random.default_rng(6)
    K, T, d_out, d_in, sigma = 3, 11, 4, 5, 0.02
    r = rng.standard_normal((K, T))
    a = orc.noise(8, 1, 2, K, T, d_out)
    g = orc.error_estimate(r, d_out, 8, 1, 2, sigma, 0)
    assert np.allclose(g, -np.einsum("kt,ktc->tc", r, a) / (K * sigma), rtol=1e-13, atol=1e-14)
    X = rng.standard_normal((T, d_in))
    assert np.allclose(orc.contract(g, X, 0.25), 0.25 * g.T @ X, rtol=1e-13, atol=1e-14)
    rows = orc.error_rows(r, d_out, [0, 5, 10], 8, 1, 2, sigma, 0)
    assert np.array_equal(rows, g[[0, 5, 10]])
    ent = orc.gW_entries(X, r, d_out, [0, 3, 2], [4, 0, 1], 8, 1, 2, sigma, 0.25, 0)
    full = orc.contract(g, X, 0.25)
    assert np.allclose(ent, full[[0, 3, 2], [4, 0, 1]], rtol=1e-13)


# ------------------------------------------------------- statistical pins --

def _planted(orc, rng, T, d_out, K, sigma, kind, seed, curv=0.0, flags=0, common=True):
    if common:
        dp = np.tile(rng.standard_normal(d_out), (T, 1))
    else:
        dp = rng.standard_normal((T, d_out))
    delta = orc.planted_delta(dp, seed, kind, 0, K, sigma, curv=curv, flags=flags)
    return dp, delta


@pytest.mark.parametrize("kind", [0, 1, 3])
@pytest.mark.parametrize("center", [False, True])
def test_unbiased_recovers_planted_error(orc, kind, center):
    """Linear loss delta = sigma <dplant, a>: E[g_t] = dplant_t without
    centring and ((K-1)/K) dplant_t with centring over the K draws."""
    rng = np.random.default_rng(10 + kind)
    T, d_out, K, sigma = 40000, 6, 4, 1e-3
    dp, delta = _planted(orc, rng, T, d_out, K, sigma, kind, seed=31)
    flags = orc.CENTER if center else 0
    r = orc.credit(delta, np.array([0, T], np.int32), 0.0, flags)
    g = orc.error_estimate(r, d_out, 31, kind, 0, sigma, flags)
    mean = g.mean(axis=0)
    want = dp[0] * ((K - 1) / K if center else 1.0)
    nrm = np.linalg.norm(dp[0])
    tol = 5.0 * nrm * np.sqrt((d_out + 2) / (T * K))
    assert np.max(np.abs(mean - want)) <= tol


def test_contraction_orientation_under_planted_loss(orc):
    """E[GW] = ((K-1)/K) sum_t dplant_t x_t^T, with d_in != d_out so that a
    transposed operand cannot pass."""
    rng = np.random.default_rng(12)
    T, d_in, d_out, K, sigma = 30000, 3, 5, 8, 1e-3
    X = rng.standard_normal((T, d_in)) + np.array([1.0, -2.0, 0.5])
    dp, delta = _planted(orc, rng, T, d_out, K, sigma, 1, seed=5)
    gW = orc.estimate_gW(X, delta, d_out, np.array([0, T], np.int32), 5, 1, 0, sigma, 0.0,
                         1.0 / T, orc.CENTER)
    want = (K - 1) / K * (dp.T @ X) / T
    assert gW.shape == (d_out, d_in)
    assert np.max(np.abs(gW - want)) <= 0.05 * np.max(np.abs(want))


@pytest.mark.parametrize("gamma", [0.0, 0.9])
def test_antithetic_cancels_even_order_term(orc, gamma):
    """With antithetic pairs the curvature term 0.5 sigma^2 |a|^2 leaves the
    estimate unchanged: the pair difference is odd in a."""
    rng = np.random.default_rng(13)
    T, d_out, K, sigma = 64, 8, 6, 0.05
    f = orc.ANTITHETIC
    dp = rng.standard_normal((T, d_out))
    lin = orc.planted_delta(dp, 17, 1, 0, K, sigma, curv=0.0, flags=f)
    quad = orc.planted_delta(dp, 17, 1, 0, K, sigma, curv=1.0, flags=f)
    assert np.max(np.abs(quad - lin)) > 1e-3
    o = np.array([0, 20, 64], np.int32)
    X = rng.standard_normal((T, 3))
    a = orc.estimate_gW(X, lin, d_out, o, 17, 1, 0, sigma, gamma, 1.0, orc.CENTER | f)
    b = orc.estimate_gW(X, quad, d_out, o, 17, 1, 0, sigma, gamma, 1.0, orc.CENTER | f)
    assert np.allclose(a, b, rtol=1e-10, atol=1e-12 * np.abs(a).max())
    # without antithetic pairs the curvature term does leak in
    lin2 = orc.planted_delta(dp, 17, 1, 0, K, sigma, curv=0.0)
    quad2 = orc.planted_delta(dp, 17, 1, 0, K, sigma, curv=1.0)
    a2 = orc.estimate_gW(X, lin2, d_out, o, 17, 1, 0, sigma, gamma, 1.0, 0)
    b2 = orc.estimate_gW(X, quad2, d_out, o, 17, 1, 0, sigma, gamma, 1.0, 0)
    assert np.max(np.abs(a2 - b2)) > 1e-3 * np.abs(a2).max()


def _cos(u, v):
    return float(np.dot(u.ravel(), v.ravel()) / (np.linalg.norm(u) * np.linalg.norm(v)))


@pytest.mark.parametrize("d,K", [(16, 16), (16, 256), (64, 64), (64, 1024)])
def test_cosine_law_per_token(orc, d, K):
    """Per-token cos(g_t, dplant_t) tracks sqrt(K / (K + D)) with D = d + 1
    for isotropic Gaussian noise (error energy (D+1)|grad|^2/K in "What a
    zeroth-order gradient is", with the per-token search dimension d_out of
    "Perturb the activations, not the weights")."""
    rng = np.random.default_rng(14)
    T, sigma = 48, 1e-3
    dp, delta = _planted(orc, rng, T, d, K, sigma, 1, seed=99, common=False)
    r = orc.credit(delta, np.array([0, T], np.int32), 0.0, 0)
    g = orc.error_estimate(r, d, 99, 1, 0, sigma, 0)
    cs = np.array([_cos(g[t], dp[t]) for t in range(T)])
    want = np.sqrt(K / (K + d + 1))
    assert abs(cs.mean() - want) <= 0.03


def _toy_rows():
    rows = []
    with open(GOLDEN_TOY) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                d, K, c = line.split()
                rows.append((int(d), int(K), float(c)))
    return rows


@pytest.mark.slow
@pytest.mark.parametrize("d,K,printed", _toy_rows())
def test_page_toy_per_token_cosine(orc, d, K, printed):
    """The page's toy: d x d layer, 32 tokens, quadratic per-token loss, K
    forward passes, one reward per token; cosine of GW to the true gradient
    sum_t delta_t x_t^T. One seeded run on the page; here the mean over a few
    seeds, within 0.015 of the printed value."""
    T, sigma = 32, 1e-3
    cs = []
    for rep in range(4):
        rng = np.random.default_rng(1000 + rep)
        X = rng.standard_normal((T, d))
        dp = rng.standard_normal((T, d))
        delta = orc.planted_delta(dp, 500 + rep, 1, 0, K, sigma, curv=1.0)
        gW = orc.estimate_gW(X, delta, d, np.array([0, T], np.int32), 500 + rep, 1, 0, sigma,
                             0.0, 1.0, 0)
        cs.append(_cos(gW, dp.T @ X))
    assert abs(np.mean(cs) - printed) <= 0.015


# ----------------------------------------------------------------- jitter --

def test_jitter_adds_sigma_times_noise(orc):
    rng = np.random.default_rng(15)
    y = rng.standard_normal((9, 13))
    out = orc.jitter(y, 3, 1, 7, 0.25)
    a = orc.noise(3, 1, 7, 1, 9, 13)[0]
    assert np.allclose(out, y + 0.25 * a, rtol=0, atol=1e-15)
