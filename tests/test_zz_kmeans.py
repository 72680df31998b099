"""GPU parity of the codebook calibration in Cholesky space (API page,
a2ats_cholesky_factor: with H = L L^T, ordinary k-means++ on the rows
z = k L trains the H-weighted codebook, and c = c_z L^-1 brings it back).

* a2ats_kmeanspp against the oracle's kmeanspp on the same fp32 rows z: the
  seeds are copies of rows of z, so they must be the oracle's bit for bit;
  the codes of every assignment equal the oracle's except on near-ties; the
  Lloyd means and the objective agree to fp32 rounding.
* a2ats_cholesky_rows and a2ats_cholesky_solve_rows against the oracle's
  change of variables and back substitution.
* The composition (rows -> k-means -> back to key space) reproduces its own
  codes under a2ats_h_weighted_assign with the same L.

The file name sorts late so a stop-at-first-failure run has run the rest of
the path's tests first.
"""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import TIE, assert_rows_close, check_codes, dev, f64

pytestmark = pytest.mark.gpu


def _draws(H, K, seed):
    return np.random.default_rng(seed).random((H, K))


def _gap(z, c):
    """Relative top-2 gap of the nearest-centroid distances (numpy, fp64,
    |z|^2 - 2 z.c + |c|^2, ample for telling a 1e-5 gap from a tie)."""
    if len(c) < 2:
        return np.full(len(z), np.inf)
    dist = (z * z).sum(1)[:, None] - 2.0 * (z @ c.T) + (c * c).sum(1)[None, :]
    dist = np.maximum(dist, 0.0)
    part = np.partition(dist, 1, axis=1)
    return (part[:, 1] - part[:, 0]) / np.maximum(part[:, 1], 1e-300)


def _run(z, K, u, iters):
    cent, codes, obj = q.a2ats_kmeanspp(dev(z), K, dev(torch.from_numpy(u)), iters)
    torch.cuda.synchronize()
    return f64(cent), codes.cpu().numpy(), obj.cpu().numpy()


@pytest.mark.parametrize("case", [
    # H, n, d, K
    (2, 300, 16, 12),
    (1, 1000, 64, 40),
    (3, 37, 8, 50),      # K > n: once every row is a centre all D^2 are 0
    (1, 2500, 128, 200),
    (2, 777, 24, 1),     # a single centre
])
def test_seeds_are_the_oracles(case):
    H, n, d, K = case
    z = synth.gaussian((H, n, d), seed=n + d, dtype="f32")
    u = _draws(H, K, seed=K)
    cent, codes, obj = _run(z, K, u, 0)
    for h in range(H):
        zh = f64(z[h])
        oc, ocodes, oobj = oracle.kmeanspp(zh, K, u[h], 0)
        np.testing.assert_array_equal(cent[h], oc)
        check_codes(codes[h], ocodes, _gap(zh, oc))
        np.testing.assert_allclose(obj[h], oobj, rtol=1e-8)


def test_duplicate_rows_and_zero_spread():
    """Rows repeated many times: the seeding reaches D^2 = 0 everywhere and
    falls back to the uniform rule, exactly like the oracle."""
    base = synth.gaussian((1, 6, 8), seed=3, dtype="f32")
    z = base[:, torch.from_numpy(np.random.default_rng(4).integers(0, 6, 400))].contiguous()
    K = 10
    u = _draws(1, K, seed=5)
    cent, codes, obj = _run(z, K, u, 3)
    oc, ocodes, oobj = oracle.kmeanspp(f64(z[0]), K, u[0], 3)
    np.testing.assert_array_equal(cent[0], oc)
    assert codes[0].tolist() == ocodes.tolist()
    np.testing.assert_allclose(obj[0], oobj, rtol=1e-12, atol=0)
    assert obj[0, -1] == 0.0


def test_lloyd_rounds_track_the_oracle():
    H, n, d, K, iters = 2, 2000, 32, 16, 6
    z = synth.gaussian((H, n, d), seed=11, dtype="f32", scale=3.0)
    u = _draws(H, K, seed=12)
    cent, codes, obj = _run(z, K, u, iters)
    for h in range(H):
        zh = f64(z[h])
        oc, ocodes, oobj = oracle.kmeanspp(zh, K, u[h], iters)
        assert_rows_close(cent[h], oc, rel=1e-6)
        check_codes(codes[h], ocodes, _gap(zh, oc))
        np.testing.assert_allclose(obj[h], oobj, rtol=1e-6)
        assert (np.diff(obj[h]) <= 1e-9 * obj[h, 0]).all()


def test_separated_blobs_are_recovered_like_the_oracle():
    K, d, per = 6, 16, 80
    rng = np.random.default_rng(21)
    centres = rng.standard_normal((K, d)) * 100.0
    truth = np.repeat(np.arange(K), per)
    zn = centres[truth] + rng.standard_normal((K * per, d))
    z = torch.from_numpy(zn[None]).to(torch.float32)
    u = _draws(1, K, seed=22)
    cent, codes, obj = _run(z, K, u, 8)
    oc, ocodes, oobj = oracle.kmeanspp(f64(z[0]), K, u[0], 8)
    assert codes[0].tolist() == ocodes.tolist()
    assert_rows_close(cent[0], oc, rel=1e-6)
    np.testing.assert_allclose(obj[0], oobj, rtol=1e-6)


def test_calibration_shape_of_the_pages():
    """Llama-3.2-3B-shaped calibration keys (one layer: 8 heads, 4096
    tokens, head_dim 128) and a 1024-entry codebook, with L = identity (the
    keys themselves as z), one Lloyd round; two heads against the oracle."""
    w = synth.scaled(synth.WORKLOADS["llama32_3b_layer"], N=4096)
    z = synth.keys(w)[0].to(torch.float32).contiguous()
    H, n, d = z.shape
    K = w.K
    u = _draws(H, K, seed=31)
    cent, codes, obj = _run(z, K, u, 1)
    for h in (0, H - 1):
        zh = f64(z[h])
        oc, ocodes, oobj = oracle.kmeanspp(zh, K, u[h], 1)
        assert_rows_close(cent[h], oc, rel=1e-6)
        check_codes(codes[h], ocodes, _gap(zh, oc))
        np.testing.assert_allclose(obj[h], oobj, rtol=1e-6)


def _spd_factor(H, d, seed):
    rng = np.random.default_rng(seed)
    Ls = []
    for _ in range(H):
        A = rng.standard_normal((d, d))
        Ls.append(oracle.cholesky(A @ A.T / d + 0.05 * np.eye(d))[0])
    return np.stack(Ls).astype(np.float32)


@pytest.mark.parametrize("dt,H,n,d", [("bf16", 2, 300, 64), ("f32", 1, 1000, 128),
                                      ("f16", 3, 17, 8)])
def test_cholesky_rows_and_solve_match_the_oracle(dt, H, n, d):
    L = _spd_factor(H, d, seed=d)
    noisy = L + np.triu(np.full((d, d), 5.0, np.float32), 1)  # ignored above the diagonal
    x = synth.gaussian((H, n, d), seed=n, dtype=dt)
    z = q.a2ats_cholesky_rows(dev(x), dev(torch.from_numpy(noisy)))
    zc = synth.gaussian((H, 40, d), seed=n + 1, dtype="f32")
    c = q.a2ats_cholesky_solve_rows(dev(zc), dev(torch.from_numpy(noisy)))
    torch.cuda.synchronize()
    for h in range(H):
        Lh = L[h].astype(np.float64)
        assert_rows_close(f64(z[h]), oracle.cholesky_rows(f64(x[h]), Lh), rel=2e-6)
        assert_rows_close(f64(c[h]), oracle.cholesky_solve_rows(f64(zc[h]), Lh), rel=1e-5)


def test_key_space_codebook_reproduces_the_codes():
    """keys -> z = k L -> k-means++ -> c = c_z L^-1: the H-weighted
    assignment of the keys with c and L gives back the k-means codes, except
    where two centroids are within rounding of each other."""
    H, n, d, K = 2, 1500, 64, 32
    L = torch.from_numpy(_spd_factor(H, d, seed=41))
    x = synth.gaussian((H, n, d), seed=42, dtype="f32")
    z = q.a2ats_cholesky_rows(dev(x), dev(L))
    u = _draws(H, K, seed=43)
    cz, codes, _ = q.a2ats_kmeanspp(z, K, dev(torch.from_numpy(u)), 4)
    c = q.a2ats_cholesky_solve_rows(cz, dev(L))
    back = q.a2ats_h_weighted_assign(dev(x).unsqueeze(0), c, dev(L))
    torch.cuda.synchronize()
    got, want = back[0].cpu().numpy(), codes.cpu().numpy()
    for h in range(H):
        zh, czh = f64(z[h]), f64(cz[h])
        differ = got[h] != want[h]
        assert (_gap(zh, czh)[differ] < 100 * TIE).all()
        assert differ.mean() < 1e-2
