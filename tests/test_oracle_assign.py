"""Pins of the oracle's H-weighted and cosine-blend assignment (CPU only).

Sources: API page, a2ats_h_weighted_assignment (Eq. 14 through the Eq. 15-18
Cholesky identity) and a2ats_query_aware_assignment (cosine blend);
deploy-preview page, Evidence list (h-weighted tests); v0.39.0 page,
Evidence list (beta tests).
"""
import numpy as np
import pytest
from scipy.spatial.distance import cdist

import oracle
from _golden import lines


def _spd(r, d, cond=30.0):
    q, _ = np.linalg.qr(r.standard_normal((d, d)))
    lam = np.exp(np.linspace(0, np.log(cond), d))
    return (q * lam) @ q.T


def test_h_weighted_assignment_matches_bruteforce_eq14():
    r = np.random.default_rng(0)
    for d, K, n in ((4, 7, 50), (16, 33, 40), (32, 64, 20)):
        x, c = r.standard_normal((n, d)), r.standard_normal((K, d))
        h = _spd(r, d)
        l, _ = oracle.cholesky(h)
        code_q, a_q, b_q = oracle.assign_quadratic(x, c, h)
        code_c, a_c, b_c = oracle.assign_cholesky(x, c, l)
        np.testing.assert_array_equal(code_q, code_c)
        np.testing.assert_allclose(a_q, a_c, rtol=1e-10)
        np.testing.assert_allclose(b_q, b_c, rtol=1e-10)


def test_quadratic_form_matches_scipy_mahalanobis():
    r = np.random.default_rng(1)
    d, K, n = 8, 19, 60
    x, c, h = r.standard_normal((n, d)), r.standard_normal((K, d)), _spd(r, d)
    D = cdist(x, c, "mahalanobis", VI=h) ** 2
    code, d1, d2 = oracle.assign_quadratic(x, c, h)
    np.testing.assert_array_equal(code, D.argmin(1))
    s = np.sort(D, 1)
    np.testing.assert_allclose(d1, s[:, 0], rtol=1e-10)
    np.testing.assert_allclose(d2, s[:, 1], rtol=1e-10)


def test_h_identity_reduces_to_plain_nearest_centroid():
    r = np.random.default_rng(2)
    d, K, n = 16, 40, 100
    x, c = r.standard_normal((n, d)), r.standard_normal((K, d))
    want = cdist(x, c, "sqeuclidean").argmin(1)
    for s in (1.0, 3.7):
        l, _ = oracle.cholesky(s * np.eye(d))
        np.testing.assert_array_equal(oracle.assign_cholesky(x, c, l)[0], want)
    np.testing.assert_array_equal(oracle.assign_cholesky(x, c, None)[0], want)


def test_h_weighted_differs_from_plain_vq_under_anisotropic_h():
    r = np.random.default_rng(3)
    d, K, n = 16, 64, 400
    x, c = r.standard_normal((n, d)), r.standard_normal((K, d))
    l, _ = oracle.cholesky(_spd(r, d, cond=1e3))
    diff = (oracle.assign_cholesky(x, c, l)[0] != oracle.assign_cholesky(x, c, None)[0]).mean()
    assert diff > 0.1


def test_exact_tie_goes_to_lowest_index():
    c = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 0.0], [0.0, 1.0]])
    x = np.array([[0.0, 0.9], [0.9, 0.0], [0.5, 0.5]])
    code, _, _ = oracle.assign_cholesky(x, c, None)
    np.testing.assert_array_equal(code, [1, 0, 0])
    assert oracle.assign_quadratic(x, c, np.eye(2))[0].tolist() == [1, 0, 0]


def test_thread_count_does_not_change_results():
    r = np.random.default_rng(4)
    x, c = r.standard_normal((97, 8)), r.standard_normal((13, 8))
    l, _ = oracle.cholesky(_spd(r, 8))
    a = oracle.assign_cholesky(x, c, l, nthreads=1)
    b = oracle.assign_cholesky(x, c, l, nthreads=7)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_beta_one_reduces_to_nearest_centroid():
    r = np.random.default_rng(5)
    d, K, n = 16, 50, 120
    x, c, q = r.standard_normal((n, d)), r.standard_normal((K, d)), r.standard_normal(d)
    code, e1, e2 = oracle.assign_blend(x, c, q, 1.0)
    D = cdist(x, c, "sqeuclidean")
    np.testing.assert_array_equal(code, D.argmin(1))
    np.testing.assert_allclose(e1, np.sort(D, 1)[:, 0], rtol=1e-12)


def test_beta_zero_is_pure_query_alignment():
    r = np.random.default_rng(6)
    d, K, n = 16, 50, 30
    x, c, q = r.standard_normal((n, d)), r.standard_normal((K, d)), r.standard_normal(d)
    want = cdist(q[None], c, "cosine").argmin()
    code, _, _ = oracle.assign_blend(x, c, q, 0.0)
    assert (code == want).all()


def test_query_aware_prefers_relevant_centroid_over_nearest():
    g = list(lines("blend_prefers_relevant.txt"))
    kv = {t[0]: t[1:] for t in g if t[0] in ("x", "query", "c")}
    x = np.array([[float(v) for v in kv["x"]]])
    q = np.array([float(v) for v in kv["query"]])
    c = np.array([float(v) for v in kv["c"]]).reshape(-1, 2)
    for t in g:
        if t[0] != "beta":
            continue
        beta, rest = float(t[1]), dict(zip(t[2::2], t[3::2]))
        code, s1, s2 = oracle.assign_blend(x, c, q, beta)
        assert code[0] == int(rest["code"])
        if "best" in rest:
            assert abs(s1[0] - float(rest["best"])) < 1e-15
            assert abs(s2[0] - float(rest["second"])) < 1e-15


def test_per_row_query_equals_shared_query_per_row():
    r = np.random.default_rng(7)
    d, K, n = 8, 21, 12
    x, c, qs = r.standard_normal((n, d)), r.standard_normal((K, d)), r.standard_normal((n, d))
    code, s1, _ = oracle.assign_blend(x, c, qs, 0.6)
    for i in range(n):
        ci, si, _ = oracle.assign_blend(x[i:i + 1], c, qs[i], 0.6)
        assert ci[0] == code[i] and si[0] == s1[i]


@pytest.mark.parametrize("beta", [0.3, 0.7])
def test_blend_scores_are_ordered_and_bounded(beta):
    r = np.random.default_rng(8)
    x, c, q = r.standard_normal((50, 8)), r.standard_normal((30, 8)), r.standard_normal(8)
    _, s1, s2 = oracle.assign_blend(x, c, q, beta)
    assert (s1 >= s2).all() and (s1 <= 1.0 + 1e-12).all() and (s2 >= -1.0 - 1e-12).all()
