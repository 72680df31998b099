"""Pins of the composed per-step path in the oracle (CPU only).

Sources: v0.39.0 page, "How it works" (split -> assignment with the
retrieval set on the query-aware rule and the bulk on plain VQ); deploy-preview
page, "Per-step re-rotation" (windowed RoPE against the current decode
position every step) and Evidence list.
"""
import numpy as np
from scipy.spatial.distance import cdist

import oracle


def _case(n=200, d=16, K=24, seed=0):
    r = np.random.default_rng(seed)
    return r.standard_normal((n, d)), r.standard_normal((K, d))


def test_bulk_rows_get_plain_vq_and_retrieval_rows_h_weighted():
    k, c = _case()
    r = np.random.default_rng(9)
    g = r.standard_normal((16, 64))
    l, _ = oracle.cholesky(g @ g.T / 64 + 1e-2 * np.eye(16))
    res = oracle.pipeline_step(k, 199, c, window=16, far_offset=0, base=10000.0,
                               fraction=0.2, l=l)
    ret, bulk = res.perm[:res.count], res.perm[res.count:]
    np.testing.assert_array_equal(res.codes[bulk],
                                  cdist(res.k_tilde[bulk], c, "sqeuclidean").argmin(1))
    h = l @ l.T
    np.testing.assert_array_equal(res.codes[ret],
                                  (cdist(res.k_tilde[ret], c, "mahalanobis", VI=h) ** 2).argmin(1))


def test_proxy_query_row_is_always_retrieved():
    k, c = _case(seed=1)
    res = oracle.pipeline_step(k, 199, c, window=8, far_offset=0, base=10000.0, fraction=0.05)
    assert 199 in res.perm[:res.count].tolist()


def test_blend_path_when_no_h():
    k, c = _case(seed=2)
    res = oracle.pipeline_step(k, 199, c, window=8, far_offset=0, base=10000.0,
                               fraction=0.1, beta=0.5)
    ret = res.perm[:res.count]
    code, _, _ = oracle.assign_blend(res.k_tilde[ret], c, res.k_tilde[199], 0.5)
    np.testing.assert_array_equal(res.codes[ret], code)


def test_token_leaves_window_as_decode_position_advances():
    k, c = _case(n=64, seed=3)
    a = oracle.pipeline_step(k[:50], 49, c, window=8, far_offset=0, base=10000.0, fraction=0.1)
    b = oracle.pipeline_step(k[:60], 59, c, window=8, far_offset=0, base=10000.0, fraction=0.1)
    assert not np.array_equal(a.k_tilde[45], k[45])
    assert np.array_equal(b.k_tilde[45], k[45])
