"""Pins of the oracle's expert similarity table (App. A.3, Eq. 6-8)."""
import numpy as np
from scipy.spatial.distance import cdist

from oracle import similarity


def test_matches_library_cosine():
    """Eq. 6 by scipy's cosine distance (1 - cos); the table is sign(cos) cos^2."""
    rng = np.random.default_rng(0)
    H = rng.standard_normal((500, 12)).astype(np.float32)
    H[:, 3] = -0.5 * H[:, 7] + 0.1 * H[:, 3]      # a strongly anti-correlated pair
    cos = 1.0 - cdist(H.T.astype(np.float64), H.T.astype(np.float64), "cosine")
    tab = similarity.table([H], 12)
    np.testing.assert_allclose(tab, np.sign(cos) * cos ** 2, rtol=1e-10, atol=1e-12)
    assert tab[3, 7] < -0.9


def test_batches_add_up():
    """Eq. 8 is accumulated over small batches: any split gives the same table."""
    rng = np.random.default_rng(1)
    H = rng.standard_normal((1000, 8))
    whole = similarity.table([H], 8)
    split = similarity.table([H[:1], H[1:333], H[333:]], 8)
    np.testing.assert_allclose(split, whole, rtol=1e-12, atol=1e-14)


def test_closed_forms():
    # orthogonal columns: 0 off the diagonal, 1 on it
    H = np.zeros((4, 3))
    H[0, 0] = 2.0
    H[1, 1] = -3.0
    H[2, 2] = 0.5
    np.testing.assert_array_equal(similarity.table([H], 3), np.eye(3))
    # a column and a negative multiple of it: -1; a zero column: 0
    H = np.array([[1.0, -2.0, 0.0], [2.0, -4.0, 0.0], [3.0, -6.0, 0.0]])
    tab = similarity.table([H], 3)
    np.testing.assert_allclose(tab[0, 1], -1.0, rtol=1e-15)
    assert (tab[2] == 0).all() and (tab[:, 2] == 0).all()
