"""GPU parity at the full sizes of the long-context and wide-head workloads,
in the launch configuration the benchmark uses (one A2ATSStep over the whole
batch), checked on sampled outputs the oracle computes one by one: H and L of
sampled heads, the whole retrieval split of sampled (sequence, head) pairs,
and the codes of sampled retrieval and bulk rows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import check_codes, check_split, dev, f64
from query_aware_vq_gb300.pipeline import A2ATSStep

pytestmark = pytest.mark.gpu


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def _run(name, pairs, n_ret, n_bulk, h_tol):
    w = synth.WORKLOADS[name]
    k, c = synth.keys(w), synth.codebook(w)
    Q = synth.queries(w) if not w.h_given else None
    Hg = synth.given_h(w) if w.h_given else None
    step = A2ATSStep(w.B, w.H, w.N, w.d, w.K, synth.DTYPES[w.dtype], window=w.W,
                     fraction=w.fraction, rope_base=w.rope_base, far_offset=w.far_offset, M=w.M,
                     ridge=w.ridge, beta=w.betas[-1])
    step(dev(k), dev(c), queries=dev(Q) if Q is not None else None,
         h_given=dev(Hg) if Hg is not None else None)
    torch.cuda.synchronize()
    assert (step.info.cpu() == 0).all()
    Lg = f64(step.L)
    codes, perm, count = step.codes.cpu().numpy(), step.perm.cpu().numpy(), step.count.cpu().numpy()
    rng = np.random.default_rng(7)
    for b, h in pairs:
        # calibration of this head, by the oracle, rounded to fp32 where the
        # pages' functions return float32 arrays
        if Q is not None:
            hm = oracle.query_second_moment(Q[h], w.ridge)
            assert _rel(f64(step.Hm[h]), hm) < 1e-6
            hm = hm.astype(np.float32).astype(np.float64)
        else:
            hm = f64(Hg[h])
        Lo, info = oracle.cholesky(hm)
        assert info == 0
        assert _rel(Lg[h], Lo) < h_tol
        Lo = Lo.astype(np.float32).astype(np.float64)
        n = w.N
        v = oracle.windowed_rope(k[b, h], np.arange(n), n - 1, w.W, w.far_offset, w.rope_base)
        _, cnt, scores, kth = oracle.select_retrieval_set(v, v[-1], w.fraction)
        check_split(perm[b, h], int(count[b, h]), n, cnt, scores, kth)
        ret, bulk = perm[b, h, :cnt], perm[b, h, cnt:n]
        ret = np.sort(rng.choice(ret, min(n_ret, len(ret)), replace=False))
        bulk = np.unique(np.concatenate([rng.choice(bulk, n_bulk, replace=False),
                                         bulk[bulk >= n - w.W]]))
        code, d1, d2 = oracle.assign_cholesky(v[ret], c[h], Lo)
        check_codes(codes[b, h, ret], code, (d2 - d1) / d2, "retrieval codes")
        code, d1, d2 = oracle.assign_cholesky(v[bulk], c[h], None)
        check_codes(codes[b, h, bulk], code, (d2 - d1) / d2, "bulk codes")


def test_llama3_8b_long_full_size_sampled():
    _run("llama3_8b_long", pairs=[(0, 0), (3, 5)], n_ret=768, n_bulk=768, h_tol=1e-5)


def test_wide_head_full_size_sampled():
    _run("wide_head", pairs=[(0, 0), (0, 17), (0, 31)], n_ret=384, n_bulk=384, h_tol=1e-3)
