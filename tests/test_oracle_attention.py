"""Pins of the oracle's code-based attention scores and top-token retrieval
(deploy-preview "A2ATS-adapted" page, "Windowed RoPE (Eq. 11-12)": far keys
unrotated with the far relative position b on the query, u = q R_b k^T;
keys inside the window with exact RoPE).  Each check comes from outside the
oracle: complex-number rotation in numpy, a hand-worked fixture, a numpy
sort."""
import numpy as np
import pytest

import oracle
from _golden import table


def _pairs(x, interleaved):
    d = x.shape[-1]
    if interleaved:
        return x[..., 0::2] + 1j * x[..., 1::2]
    return x[..., : d // 2] + 1j * x[..., d // 2:]


def _rel_score(q, k, rel, base, interleaved=False):
    """RoPE(q, p + rel) . RoPE(k, p) for any p, as complex pairs: the dot of
    two rotated 2-vectors is Re(z1 conj(z2)) and rotations compose."""
    d = q.shape[-1]
    theta = base ** (-2.0 * np.arange(d // 2) / d)
    zq = _pairs(q, interleaved) * np.exp(1j * rel * theta)
    return np.real(zq[None, :] * np.conj(_pairs(k, interleaved))).sum(-1)


@pytest.mark.parametrize("interleaved", [False, True])
def test_all_near_is_exact_rope_attention(interleaved):
    rng = np.random.default_rng(1)
    n, d, base = 40, 16, 500.0
    k, q = rng.standard_normal((n, d)), rng.standard_normal(d)
    t = n - 1
    _, _, s, _ = oracle.code_attention_topk(k, t, np.zeros(n, np.int32), np.zeros((1, d)), q,
                                            window=n, far_b=7.0, base=base, fraction=0.1,
                                            interleaved=interleaved)
    want = np.array([_rel_score(q, k[j:j + 1], t - j, base, interleaved)[0] for j in range(n)])
    np.testing.assert_allclose(s, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("interleaved", [False, True])
def test_far_rows_score_their_centroid_at_relative_position_b(interleaved):
    rng = np.random.default_rng(2)
    n, d, K, base, b = 50, 8, 6, 1e4, 2048.0
    k, q = rng.standard_normal((n, d)), rng.standard_normal(d)
    c = rng.standard_normal((K, d))
    codes = rng.integers(0, K, n).astype(np.int32)
    _, _, s, _ = oracle.code_attention_topk(k, n - 1, codes, c, q, window=0, far_b=b, base=base,
                                            fraction=0.2, interleaved=interleaved)
    np.testing.assert_allclose(s, _rel_score(q, c[codes], b, base, interleaved), rtol=1e-12,
                               atol=1e-12)
    # the codebook holding the keys themselves gives the exact far score
    _, _, s2, _ = oracle.code_attention_topk(k, n - 1, np.arange(n, dtype=np.int32), k, q,
                                             window=0, far_b=b, base=base, fraction=0.2,
                                             interleaved=interleaved)
    np.testing.assert_allclose(s2, _rel_score(q, k, b, base, interleaved), rtol=1e-12,
                               atol=1e-12)


def test_window_splits_rows_by_distance_to_t():
    rng = np.random.default_rng(3)
    n, d, K, base, b, W = 64, 8, 5, 1e4, 100.0, 10
    k, q, c = rng.standard_normal((n, d)), rng.standard_normal(d), rng.standard_normal((K, d))
    codes = rng.integers(0, K, n).astype(np.int32)
    t = 55  # rows past t count as far (t - j < 0), as the windowed RoPE does
    _, _, s, _ = oracle.code_attention_topk(k, t, codes, c, q, window=W, far_b=b, base=base,
                                            fraction=0.3)
    near = (t - np.arange(n) >= 0) & (t - np.arange(n) < W)
    far_want = _rel_score(q, c[codes], b, base)
    near_want = np.array([_rel_score(q, k[j:j + 1], t - j, base)[0] for j in range(n)])
    np.testing.assert_allclose(s, np.where(near, near_want, far_want), rtol=1e-12, atol=1e-12)


def test_far_query_rotation_does_not_depend_on_the_window():
    """The far relative position b rides on the query whatever the window
    (deploy-preview page, Eq. 11): rows that are far under two windows score
    the same under both, and equal the score at relative position b."""
    rng = np.random.default_rng(5)
    n, d, K, base, b = 80, 8, 6, 1e4, 2048.0
    k, q, c = rng.standard_normal((n, d)), rng.standard_normal(d), rng.standard_normal((K, d))
    codes = rng.integers(0, K, n).astype(np.int32)
    t = n - 1
    _, _, s4, _ = oracle.code_attention_topk(k, t, codes, c, q, window=4, far_b=b, base=base,
                                             fraction=0.2)
    _, _, s40, _ = oracle.code_attention_topk(k, t, codes, c, q, window=40, far_b=b,
                                              base=base, fraction=0.2)
    far_both = t - np.arange(n) >= 40
    np.testing.assert_array_equal(s4[far_both], s40[far_both])
    np.testing.assert_allclose(s4[far_both], _rel_score(q, c[codes[far_both]], b, base),
                               rtol=1e-12, atol=1e-12)


def test_out_of_range_codes_score_zero():
    rng = np.random.default_rng(4)
    n, d = 6, 4
    codes = np.array([0, -1, 3, 1, 99, 2], np.int32)
    _, _, s, _ = oracle.code_attention_topk(rng.standard_normal((n, d)), n - 1, codes,
                                            rng.standard_normal((3, d)), rng.standard_normal(d),
                                            window=0, far_b=1.0, base=100.0, fraction=0.5)
    assert s[1] == 0.0 and s[2] == 0.0 and s[4] == 0.0


@pytest.mark.parametrize("fraction", [0.0, 0.07, 0.5, 1.0])
def test_top_tokens_follow_score_then_index(fraction):
    rng = np.random.default_rng(5)
    n, d, K = 200, 8, 4  # few centroids: many equal far scores, ties by index
    k, q, c = rng.standard_normal((n, d)), rng.standard_normal(d), rng.standard_normal((K, d))
    codes = rng.integers(0, K, n).astype(np.int32)
    perm, count, s, kth = oracle.code_attention_topk(k, n - 1, codes, c, q, window=16,
                                                     far_b=64.0, base=1e4, fraction=fraction)
    order = np.lexsort((np.arange(n), -s))
    assert count == oracle.retrieval_count(fraction, n)
    assert perm[:count].tolist() == sorted(order[:count].tolist())
    assert perm[count:].tolist() == sorted(order[count:].tolist())
    if count:
        assert kth == s[order[count - 1]]


def test_hand_worked_fixture():
    g = table("code_attention_d2.txt")
    f = lambda key: [float(v) for v in g[key][0]]
    d = int(f("d")[0])
    keys = np.array(f("keys")).reshape(-1, d)
    perm, count, s, _ = oracle.code_attention_topk(
        keys, int(f("t")[0]), np.array(f("codes"), np.int32), np.array(f("codebook")).reshape(-1, d),
        np.array(f("q")), window=int(f("window")[0]), far_b=f("far_b")[0], base=f("base")[0],
        fraction=f("fraction")[0])
    np.testing.assert_allclose(s, f("scores"), rtol=0, atol=1e-15)
    assert count == int(f("count")[0])
    assert perm.tolist() == [int(v) for v in f("perm")]
