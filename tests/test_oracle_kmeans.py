"""Pins of the oracle's codebook calibration in z space (API page,
a2ats_cholesky_factor: after z = k L with H = L L^T, ordinary squared
distances between z rows are the H-weighted ones, so ordinary k-means++ on
the z rows trains the codebook): k-means++ seeding with given uniform draws,
then Lloyd rounds."""
import numpy as np
import pytest

import oracle
from _golden import table


@pytest.mark.parametrize("name", ["kmeanspp_1d.txt", "kmeanspp_1d_offset.txt",
                                  "kmeanspp_1d_empty.txt"])
def test_hand_worked_fixture(name):
    g = table(name)
    f = lambda k: [float(v) for v in g[k][0]]
    u = np.array(f("u"))
    cent, codes, obj = oracle.kmeanspp(np.array(f("points"))[:, None], len(u), u,
                                       int(f("iters")[0]))
    np.testing.assert_array_equal(cent[:, 0], f("centroids"))
    assert codes.tolist() == [int(v) for v in f("codes")]
    np.testing.assert_array_equal(obj, f("objective"))


def test_lloyd_never_raises_the_objective():
    rng = np.random.default_rng(0)
    z = rng.standard_normal((500, 6))
    _, _, obj = oracle.kmeanspp(z, 12, rng.random(12), 15)
    assert (np.diff(obj) <= 1e-9 * obj[0]).all()


def test_separated_blobs_are_recovered():
    rng = np.random.default_rng(1)
    K, d, per = 5, 4, 60
    centres = rng.standard_normal((K, d)) * 100.0
    truth = np.repeat(np.arange(K), per)
    z = centres[truth] + rng.standard_normal((K * per, d))
    cent, codes, _ = oracle.kmeanspp(z, K, rng.random(K), 10)
    # each found cluster is one true blob, and its centroid is the blob's mean
    for j in range(K):
        members = truth[codes == j]
        assert members.size == per and (members == members[0]).all()
        np.testing.assert_allclose(cent[j], z[codes == j].mean(0), rtol=0, atol=1e-9)


def test_one_centre_per_point_gives_zero_objective():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((30, 3))
    cent, codes, obj = oracle.kmeanspp(z, 30, rng.random(30), 2)
    assert obj[-1] == 0.0
    assert sorted(codes.tolist()) == list(range(30))


def test_assignment_step_is_the_plain_nearest_centroid():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((200, 8))
    cent, codes, _ = oracle.kmeanspp(z, 16, rng.random(16), 3)
    want, _, _ = oracle.assign_cholesky(z, cent, None)
    assert codes.tolist() == want.tolist()


def test_codebook_in_key_space_reaches_the_h_weighted_rule():
    """With c = c_z L^-1 the key-space codebook's H-weighted codes of the
    keys are the z-space nearest-centroid codes (API page, Eq. 16-18)."""
    rng = np.random.default_rng(4)
    d, n, K = 8, 300, 10
    A = rng.standard_normal((d, d))
    hm = A @ A.T / d + 0.1 * np.eye(d)
    L = np.linalg.cholesky(hm)
    k = rng.standard_normal((n, d))
    z = k @ L
    cz, codes, _ = oracle.kmeanspp(z, K, rng.random(K), 5)
    c = np.linalg.solve(L.T, cz.T).T  # c L = c_z
    want, _, _ = oracle.assign_cholesky(k, c, L)
    assert want.tolist() == codes.tolist()


def test_cholesky_rows_hand_worked():
    # x = (1, 2), L = [[2, 0], [3, 4]]: z_0 = 1*2 + 2*3 = 8, z_1 = 2*4 = 8
    l = np.array([[2.0, 0.0], [3.0, 4.0]])
    z = oracle.cholesky_rows(np.array([[1.0, 2.0]]), l)
    np.testing.assert_array_equal(z, [[8.0, 8.0]])
    # back: c_1 = 8 / 4 = 2, c_0 = (8 - 2 * 3) / 2 = 1
    np.testing.assert_array_equal(oracle.cholesky_solve_rows(z, l), [[1.0, 2.0]])


def test_cholesky_rows_give_the_h_weighted_norm():
    """|x L|^2 = x H x^T with H = L L^T (the identity behind the route)."""
    rng = np.random.default_rng(5)
    d = 12
    A = rng.standard_normal((d, d))
    hm = A @ A.T / d + 0.2 * np.eye(d)
    L = np.linalg.cholesky(hm)
    x = rng.standard_normal((40, d))
    z = oracle.cholesky_rows(x, L)
    np.testing.assert_allclose((z * z).sum(1), np.einsum("na,ab,nb->n", x, hm, x), rtol=1e-12)
    np.testing.assert_array_equal(oracle.cholesky_rows(x, np.eye(d)), x)


def test_cholesky_solve_rows_is_the_triangular_solve():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(6)
    d = 16
    A = rng.standard_normal((d, d))
    L = np.linalg.cholesky(A @ A.T / d + 0.1 * np.eye(d))
    z = rng.standard_normal((25, d))
    want = scipy_linalg.solve_triangular(L.T, z.T, lower=False).T
    np.testing.assert_allclose(oracle.cholesky_solve_rows(z, L), want, rtol=1e-10, atol=1e-12)
