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


def _rotate(x, pos, base):
    """RoPE of the rows of x at positions pos as complex multiplication
    (half-split pairs (i, i + d/2), frequency base^(-2i/d))."""
    d = x.shape[1]
    h = d // 2
    w = base ** (-2.0 * np.arange(h) / d)
    z = (x[:, :h] + 1j * x[:, h:]) * np.exp(1j * np.asarray(pos, float)[:, None] * w)
    return np.concatenate([z.real, z.imag], axis=1)


def test_far_rows_of_the_step_take_the_shared_far_rotation():
    """With far_offset = b the step's far rows are every key rotated at b,
    the window rows at their own positions, and the bulk codes are the plain
    nearest centroid of those rows (deploy-preview page, Eq. 11-12)."""
    k, c = _case(n=120, seed=4)
    t, W, b = 119, 10, 37
    res = oracle.pipeline_step(k, t, c, window=W, far_offset=b, base=10000.0, fraction=0.1)
    pos = np.where(t - np.arange(120) < W, np.arange(120), b)
    np.testing.assert_allclose(res.k_tilde, _rotate(k, pos, 10000.0), rtol=0, atol=1e-12)
    bulk = res.perm[res.count:]
    np.testing.assert_array_equal(res.codes[bulk],
                                  cdist(res.k_tilde[bulk], c, "sqeuclidean").argmin(1))
