"""Pins for the oracle's embedding reassembly ("Dust: every token is a member
of the population", "What the released code actually does", step 7: the
error estimate becomes a weight gradient by "a scatter-add for an
embedding"): gE[v] = scale * sum over tokens with id v of g_t."""
import numpy as np


def test_matches_an_independent_scatter(orc):
    """Against numpy's unbuffered np.add.at (another routine)."""
    rng = np.random.default_rng(1)
    T, d, V = 500, 17, 40
    g = rng.standard_normal((T, d))
    ids = rng.integers(0, V, T).astype(np.int32)
    got, bad = orc.scatter_gE(g, ids, V, 0.25)
    want = np.zeros((V, d))
    np.add.at(want, ids, g)
    assert bad == 0
    assert np.allclose(got, 0.25 * want, rtol=1e-13, atol=1e-13)


def test_mass_is_conserved_and_unused_rows_are_zero(orc):
    rng = np.random.default_rng(2)
    T, d, V = 300, 8, 1000
    g = rng.standard_normal((T, d))
    ids = rng.integers(0, 50, T).astype(np.int32)  # rows 50.. never hit
    got, _ = orc.scatter_gE(g, ids, V)
    assert np.allclose(got.sum(axis=0), g.sum(axis=0), rtol=1e-12, atol=1e-12)
    assert np.count_nonzero(got[50:]) == 0


def test_one_id_sums_every_row_and_distinct_ids_permute(orc):
    rng = np.random.default_rng(3)
    T, d = 64, 5
    g = rng.standard_normal((T, d))
    same, _ = orc.scatter_gE(g, np.full(T, 3, np.int32), 4)
    assert np.allclose(same[3], g.sum(axis=0), rtol=1e-12)
    perm = rng.permutation(T).astype(np.int32)
    out, _ = orc.scatter_gE(g, perm, T)
    assert np.array_equal(out[perm], g)


def test_out_of_range_ids_are_skipped_and_counted(orc):
    g = np.ones((5, 2))
    out, bad = orc.scatter_gE(g, np.array([0, -1, 2, 3, 7], np.int32), 3)
    assert bad == 3
    assert np.array_equal(out, np.array([[1.0, 1.0], [0.0, 0.0], [1.0, 1.0]]))
