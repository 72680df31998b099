"""GPU parity: query second moment and Cholesky factor against the oracle
(API page, a2ats_query_second_moment / a2ats_cholesky_factor; Eq. 10, 15)."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import dev, f64

pytestmark = pytest.mark.gpu


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("H,M,d,dt", [(2, 1000, 128, "bf16"), (1, 33, 8, "f32"), (3, 517, 24, "f16"),
                                      (1, 4096, 256, "bf16"), (2, 1, 64, "f32"),
                                      # the tensor-core path: fp16, ragged slices; and the longest
                                      # slices it takes (512 rows per accumulator)
                                      (2, 3000, 128, "f16"), (1, 131072, 128, "bf16"),
                                      (1, 100, 128, "bf16")])
def test_second_moment_matches_oracle(H, M, d, dt):
    Q = synth.gaussian((H, M, d), seed=M + d, dtype=dt, scale=2.0)
    got = q.a2ats_query_second_moment(dev(Q), 1e-4)
    g = f64(got)
    for h in range(H):
        want = oracle.query_second_moment(Q[h], 1e-4)
        assert _rel(g[h], want) < 1e-6
        assert np.array_equal(g[h], g[h].T)


@pytest.mark.parametrize("name", ["llama32_3b_layer"])
def test_second_moment_full_size(name):
    w = synth.WORKLOADS[name]
    Q = synth.queries(w)
    g = f64(q.a2ats_query_second_moment(dev(Q), w.ridge))
    for h in range(w.H):
        assert _rel(g[h], oracle.query_second_moment(Q[h], w.ridge)) < 1e-6


def _spd(rng, d, cond):
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    lam = np.exp(np.linspace(0, np.log(cond), d))
    return ((Qm * lam) @ Qm.T).astype(np.float32)


@pytest.mark.parametrize("d,cond", [(8, 10.0), (16, 1e3), (128, 10.0), (256, 1e2)])
def test_cholesky_matches_oracle(d, cond):
    rng = np.random.default_rng(d)
    Hs = np.stack([_spd(rng, d, cond) for _ in range(3)])
    L, info = q.a2ats_cholesky_factor(dev(torch.from_numpy(Hs)))
    assert info.cpu().tolist() == [0, 0, 0]
    g = f64(L)
    for h in range(3):
        want, inf = oracle.cholesky(Hs[h].astype(np.float64))
        assert inf == 0
        assert _rel(g[h], want) < 1e-5
        assert np.array_equal(g[h], np.tril(g[h]))


def test_cholesky_ill_conditioned_wide_heads():
    w = synth.WORKLOADS["wide_head"]
    Hs = synth.given_h(w)
    L, info = q.a2ats_cholesky_factor(dev(Hs))
    assert (info.cpu() == 0).all()
    g = f64(L)
    for h in range(w.H):
        want, inf = oracle.cholesky(f64(Hs[h]))
        assert inf == 0
        assert _rel(g[h], want) < 1e-3


def test_cholesky_reports_non_pd_head():
    rng = np.random.default_rng(1)
    Hs = np.stack([_spd(rng, 16, 10.0) for _ in range(3)])
    Hs[1][5, 5] = -3.0   # breaks positive definiteness at or before minor 6
    L, info = q.a2ats_cholesky_factor(dev(torch.from_numpy(Hs)))
    want = [oracle.cholesky(Hs[h].astype(np.float64))[1] for h in range(3)]
    assert info.cpu().tolist() == want
    assert want[0] == 0 and want[1] > 0
