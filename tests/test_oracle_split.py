"""Pins of the oracle's retrieval split (CPU only).

Source: API page, a2ats_select_retrieval_set (top ceil(fraction * N) tokens by
key-query cosine; disjoint index sets covering 0..N-1); v0.39.0 page, Evidence
list (test_retrieval_set_picks_most_similar_to_query).
"""
import numpy as np
from scipy.spatial.distance import cdist

import oracle
from _golden import lines, table


def test_sizes_are_ceil_fraction_n():
    for f, n, k in lines("retrieval_sizes.txt"):
        f, n, k = float(f), int(n), int(k)
        assert oracle.retrieval_count(f, n) == k
        if n <= 65536:
            keys = np.random.default_rng(n).standard_normal((n, 4))
            perm, count, _, _ = oracle.select_retrieval_set(keys, np.ones(4), f)
            assert count == k


def test_retrieval_set_picks_most_similar_to_query():
    g = table("retrieval_ranking.txt")
    phi = np.radians([float(v) for v in g["phi"][0]])
    rad = np.array([float(v) for v in g["r"][0]])
    keys = np.stack([rad * np.cos(phi), rad * np.sin(phi)], 1)
    perm, count, _, _ = oracle.select_retrieval_set(keys, np.array([1.0, 0.0]),
                                                    float(g["fraction"][0][0]))
    assert perm[:count].tolist() == [int(v) for v in g["retrieval"][0]]
    assert perm[count:].tolist() == [int(v) for v in g["bulk"][0]]


def test_partition_is_disjoint_covering_and_sorted():
    r = np.random.default_rng(3)
    for n, f in ((1, 0.5), (17, 0.2), (500, 0.05), (500, 1.0), (500, 0.0)):
        keys, q = r.standard_normal((n, 8)), r.standard_normal(8)
        perm, count, _, _ = oracle.select_retrieval_set(keys, q, f)
        assert sorted(perm.tolist()) == list(range(n))
        assert perm[:count].tolist() == sorted(perm[:count].tolist())
        assert perm[count:].tolist() == sorted(perm[count:].tolist())


def test_matches_library_sort_of_cosines():
    r = np.random.default_rng(4)
    n, d, f = 300, 16, 0.13
    keys, q = r.standard_normal((n, d)), r.standard_normal(d)
    s = 1.0 - cdist(keys, q[None], "cosine")[:, 0]
    order = np.lexsort((np.arange(n), -s))
    k = oracle.retrieval_count(f, n)
    perm, count, scores, kth = oracle.select_retrieval_set(keys, q, f)
    assert count == k
    assert perm[:count].tolist() == sorted(order[:k].tolist())
    np.testing.assert_allclose(scores, s, atol=1e-12)
    assert abs(kth - s[order[k - 1]]) < 1e-12


def test_equal_scores_keep_lower_index():
    keys = np.array([[1.0, 0.0]] * 6)
    perm, count, _, _ = oracle.select_retrieval_set(keys, np.array([1.0, 0.0]), 0.5)
    assert perm[:count].tolist() == [0, 1, 2]


def test_zero_norm_key_scores_zero():
    keys = np.array([[0.0, 0.0], [1.0, 0.0], [-1.0, 0.0]])
    perm, count, scores, _ = oracle.select_retrieval_set(keys, np.array([1.0, 0.0]), 0.5)
    assert scores.tolist() == [0.0, 1.0, -1.0]
    assert perm[:count].tolist() == [0, 1]
