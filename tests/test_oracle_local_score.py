"""Pins for the oracle's local score ("Dust: every token is a member of the
population", "What the released code actually does", step 4): the score of a
jittered draw at token s is c_s = -<g_s, delta_o_s>, the estimated output
error against the block output's change; the oracle returns the loss change
delta = <g_s, delta_o_s> whose reduction is c_s."""
import numpy as np


def test_output_change_along_the_error_scores_its_squared_norm(orc):
    """delta_o_s = alpha_k g_s gives delta[k][s] = alpha_k |g_s|^2."""
    rng = np.random.default_rng(1)
    T, d, K = 50, 33, 4
    g = rng.standard_normal((T, d))
    alpha = np.array([0.5, -2.0, 0.0, 3.25])
    delta_o = alpha[:, None, None] * g[None]
    got = orc.local_score(g, delta_o)
    want = alpha[:, None] * np.sum(g * g, axis=1)[None]
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)


def test_orthogonal_change_scores_zero(orc):
    rng = np.random.default_rng(2)
    T, d, K = 20, 16, 3
    g = rng.standard_normal((T, d))
    v = rng.standard_normal((K, T, d))
    # remove each row's component along g_s
    proj = np.sum(v * g[None], axis=2) / np.sum(g * g, axis=1)[None]
    v -= proj[..., None] * g[None]
    assert np.max(np.abs(orc.local_score(g, v))) <= 1e-12


def test_matches_an_independent_contraction(orc):
    """Against numpy's einsum (another routine) on random data, with a
    one-channel and a one-token case."""
    rng = np.random.default_rng(3)
    for T, d, K in ((37, 129, 5), (1, 8, 2), (10, 1, 3)):
        g = rng.standard_normal((T, d))
        v = rng.standard_normal((K, T, d))
        assert np.allclose(orc.local_score(g, v), np.einsum("sd,ksd->ks", g, v),
                           rtol=1e-12, atol=1e-12)


def test_feeds_the_scan_as_a_loss_change(orc):
    """Keys and values sum the later tokens' scores decayed by gamma: through
    the scan, a block whose output change is the error itself at one token
    credits every earlier token of its sequence with gamma^(s-t) times the
    score's reduction."""
    T, d = 6, 4
    g = np.zeros((T, d))
    g[4] = [1.0, 2.0, 0.0, -1.0]
    delta_o = g[None].copy()  # one draw, change = error
    delta = orc.local_score(g, delta_o)
    assert delta[0, 4] == 6.0
    r = orc.credit(delta, np.array([0, T], np.int32), 0.98, 0)
    want = np.array([-6.0 * 0.98 ** (4 - t) if t <= 4 else 0.0 for t in range(T)])
    assert np.allclose(r[0], want, rtol=1e-14, atol=1e-14)
