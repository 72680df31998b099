"""Pins of the oracle's query second moment and Cholesky factor (CPU only).

Sources: API page, a2ats_query_second_moment (H = E[q^T q] + ridge I,
paper Eq. 10) and a2ats_cholesky_factor (H = L L^T, Eq. 15).
"""
import math

import numpy as np

import oracle
import synth
from _golden import table


def test_second_moment_brute_force_loops():
    r = np.random.default_rng(0)
    M, d, ridge = 5, 3, 0.25
    q = r.standard_normal((M, d))
    h = oracle.query_second_moment(q, ridge)
    for a in range(d):
        for b in range(d):
            s = 0.0
            for m in range(M):
                s += q[m][a] * q[m][b]
            want = s / M + (ridge if a == b else 0.0)
            assert abs(h[a, b] - want) < 1e-14


def test_second_moment_single_query_is_outer_product():
    q = np.array([[1.0, -2.0, 3.0]])
    h = oracle.query_second_moment(q, 1e-4)
    np.testing.assert_array_equal(h, np.outer(q[0], q[0]) + 1e-4 * np.eye(3))


def test_second_moment_is_exactly_symmetric():
    q = np.random.default_rng(1).standard_normal((300, 16))
    h = oracle.query_second_moment(q, 1e-4)
    assert np.array_equal(h, h.T)


def test_second_moment_converges_to_generator_covariance():
    # the generator's queries have covariance A A^T / d + 0.5 I (closed form)
    w = synth.scaled(synth.WORKLOADS["tiny"], d=16, H=1, M=200000, dtype="f32")
    q = synth.queries(w)[0]
    A, _ = synth._outliers_and_mixing(0, w.d)
    sigma = A @ A.T / w.d + 0.5 * np.eye(w.d)
    h = oracle.query_second_moment(q, 0.0)
    rel = np.linalg.norm(h - sigma) / np.linalg.norm(sigma)
    assert rel < 0.02


def test_cholesky_golden_integer_factor():
    g = table("cholesky_3x3.txt")
    H = np.array([float(v) for v in g["H"][0]]).reshape(3, 3)
    want = np.array([float(v) for v in g["L"][0]]).reshape(3, 3)
    l, info = oracle.cholesky(H)
    assert info == 0
    np.testing.assert_allclose(l, want, atol=1e-14)


def test_cholesky_two_by_two_closed_form():
    l, info = oracle.cholesky(np.array([[4.0, 2.0], [2.0, 3.0]]))
    assert info == 0
    np.testing.assert_allclose(l, [[2.0, 0.0], [1.0, math.sqrt(2.0)]], atol=1e-15)


def test_cholesky_matches_numpy_and_reconstructs():
    r = np.random.default_rng(2)
    for d in (1, 7, 32, 128):
        g = r.standard_normal((d, 2 * d))
        h = g @ g.T / (2 * d) + 1e-3 * np.eye(d)
        l, info = oracle.cholesky(h)
        assert info == 0
        assert np.array_equal(l, np.tril(l))
        np.testing.assert_allclose(l, np.linalg.cholesky(h), rtol=1e-10, atol=1e-12)
        assert np.linalg.norm(l @ l.T - h) <= 1e-12 * np.linalg.norm(h)


def test_cholesky_reports_first_non_pd_minor():
    assert oracle.cholesky(np.array([[-1.0]]))[1] == 1
    assert oracle.cholesky(np.zeros((3, 3)))[1] == 1
    assert oracle.cholesky(np.array([[1.0, 2.0], [2.0, 1.0]]))[1] == 2
    h = np.eye(4)
    h[2, 2] = -5
    assert oracle.cholesky(h)[1] == 3
