"""Pins of the oracle's windowed RoPE (CPU only).

Sources: deploy-preview "A2ATS-adapted" page, paper-fidelity section
(Eq. 11-12) and its Evidence list; v0.39.0 page, "How it works" step 4 and
Evidence list.
"""
import numpy as np
import pytest

import oracle
from _golden import table

pytestmark = pytest.mark.filterwarnings("ignore")


def _rng(s=0):
    return np.random.default_rng(s)


def test_golden_d4_closed_form():
    g = table("rope_d4.txt")
    x = np.array([float(v) for v in g["x"][0]])
    want = np.array([float(v) for v in g["y"][0]])
    got = oracle.rope_row(x, float(g["pos"][0][0]), float(g["base"][0][0]))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


@pytest.mark.parametrize("interleaved", [False, True])
def test_matches_complex_multiplication(interleaved):
    # RoPE is multiplication of each pair, read as a complex number, by
    # exp(i * theta_i): an independent formulation through numpy's complex exp.
    d, base = 16, 10000.0
    x = _rng(1).standard_normal(d)
    for pos in (0.0, 1.0, 7.0, 1234.0, 131071.0):
        if interleaved:
            a, b = x[0::2], x[1::2]
        else:
            a, b = x[: d // 2], x[d // 2:]
        theta = pos * base ** (-np.arange(0, d, 2) / d)
        z = (a + 1j * b) * np.exp(1j * theta)
        want = np.empty(d)
        if interleaved:
            want[0::2], want[1::2] = z.real, z.imag
        else:
            want[: d // 2], want[d // 2:] = z.real, z.imag
        got = oracle.rope_row(x, pos, base, interleaved)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_norm_preserved_per_pair():
    d = 32
    x = _rng(2).standard_normal(d)
    y = oracle.rope_row(x, 4321.0, 500000.0)
    np.testing.assert_allclose(x[:16] ** 2 + x[16:] ** 2, y[:16] ** 2 + y[16:] ** 2, rtol=1e-13)


def test_relative_position_identity():
    # <R(q, i), R(k, j)> = <R(q, i - j), k>: attention depends on i - j only.
    d, base = 64, 500000.0
    r = _rng(3)
    q, k = r.standard_normal(d), r.standard_normal(d)
    for i, j in ((10, 3), (1000, 999), (65536, 17)):
        lhs = oracle.rope_row(q, i, base) @ oracle.rope_row(k, j, base)
        rhs = oracle.rope_row(q, i - j, base) @ k
        assert abs(lhs - rhs) < 1e-9 * (np.abs(q).sum() * np.abs(k).sum())


def test_position_zero_is_identity():
    x = _rng(4).standard_normal(128)
    assert np.array_equal(oracle.rope_row(x, 0.0, 500000.0), x)


def _win(x, t, W, far=0, base=500000.0):
    n = x.shape[0]
    return oracle.windowed_rope(x, np.arange(n), t, W, far, base)


def test_windowed_rope_within_window_matches_exact_rope():
    n, d, W = 50, 16, 8
    x = _rng(5).standard_normal((n, d))
    t = n - 1
    y = _win(x, t, W)
    for p in range(t - W + 1, t + 1):
        assert np.array_equal(y[p], oracle.rope_row(x[p], p, 500000.0))


def test_windowed_rope_outside_window_returns_key_unrotated():
    n, d, W = 50, 16, 8
    x = _rng(6).standard_normal((n, d))
    y = _win(x, n - 1, W)
    assert np.array_equal(y[: n - W], x[: n - W])
    assert not np.allclose(y[n - W:], x[n - W:])


def test_window_boundary_is_exactly_w_rows():
    n, d, W = 40, 8, 5
    x = _rng(7).standard_normal((n, d))
    y = _win(x, n - 1, W)
    changed = [p for p in range(n) if not np.array_equal(y[p], x[p])]
    assert changed == list(range(n - W, n))


def test_far_tokens_are_position_independent():
    n, d, W, far = 30, 16, 4, 37
    row = _rng(8).standard_normal(d)
    x = np.tile(row, (n, 1))
    y = _win(x, n - 1, W, far=far)
    for p in range(n - W):
        assert np.array_equal(y[p], y[0])
    assert np.array_equal(y[0], oracle.rope_row(row, far, 500000.0))


def test_window_zero_always_unrotated():
    x = _rng(9).standard_normal((20, 8))
    for W in (0, -3):
        assert np.array_equal(_win(x, 19, W), x)


def test_window_exceeds_seqlen_always_exact():
    n = 20
    x = _rng(10).standard_normal((n, 8))
    for W in (n, n + 1, 10 ** 6):
        y = _win(x, n - 1, W)
        for p in range(n):
            assert np.array_equal(y[p], oracle.rope_row(x[p], p, 500000.0))


def test_token_rotation_updates_as_decode_position_advances():
    n, d, W = 64, 16, 8
    x = _rng(11).standard_normal((n, d))
    p = 40
    y_near = oracle.windowed_rope(x[p:p + 1], [p], 45, W, 0, 500000.0)
    y_far = oracle.windowed_rope(x[p:p + 1], [p], 48, W, 0, 500000.0)
    assert np.array_equal(y_near[0], oracle.rope_row(x[p], p, 500000.0))
    assert np.array_equal(y_far[0], x[p])
