"""Pins for the oracle's jittered forward (y = X W^T, then y + sigma a_t for
each draw: "Dust: every token is a member of the population", "Perturb the
activations, not the weights")."""
import numpy as np


def test_clean_slice_is_the_product(orc):
    rng = np.random.default_rng(1)
    X = rng.standard_normal((37, 19))
    W = rng.standard_normal((23, 19))
    out = orc.forward_jitter(X, W, 3, orc.GAUSSIAN, 0, 2, 0.5, clean=True)
    assert out.shape == (3, 37, 23)
    assert np.allclose(out[0], X @ W.T, rtol=1e-13, atol=1e-13)


def test_draw_slices_are_the_product_plus_the_jitter(orc):
    """Each draw's slice is the clean product with the oracle's own jitter
    applied (an independent entry point), for every noise kind and with
    antithetic pairs."""
    rng = np.random.default_rng(2)
    X = rng.standard_normal((40, 8))
    W = rng.standard_normal((70, 8))
    y = X @ W.T
    for kind in (0, 1, 3):
        for flags in (0, orc.ANTITHETIC):
            out = orc.forward_jitter(X, W, 9, kind, 4, 3, 0.25, flags)
            for k in range(3):
                want = orc.jitter(y, 9, kind, 4 + k, 0.25, flags)
                assert np.allclose(out[k], want, rtol=1e-13, atol=1e-13)


def test_zero_sigma_repeats_the_product(orc):
    rng = np.random.default_rng(3)
    X = rng.standard_normal((5, 4))
    W = rng.standard_normal((6, 4))
    out = orc.forward_jitter(X, W, 1, orc.GAUSSIAN, 0, 4, 0.0)
    for k in range(4):
        assert np.array_equal(out[k], out[0])
