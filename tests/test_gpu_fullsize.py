"""GPU parity at the full sizes of the long-context and wide-head workloads,
in the launch configuration the benchmark uses (one A2ATSStep over the whole
batch), checked on outputs the oracle computes one by one: the whole
retrieval split of every (sequence, head) and the codes of a few of its
retrieval and bulk rows; H and L of sampled heads and the codes of many
rows of sampled pairs; and the rotated keys: every RoPE-window row of every
(sequence, head) in the storage format, and rows at the highest positions
(up to 131071) rotated exactly in fp32 (deploy-preview page "A2ATS-adapted",
"Windowed RoPE (Eq. 11-12)")."""
import numpy as np
import pytest
import torch

import oracle
import synth
import query_aware_vq_gb300 as q
from _parity import (assert_rows_close, assert_storage_close, check_codes, check_split,
                     dev, f64)
from query_aware_vq_gb300.pipeline import A2ATSStep

pytestmark = pytest.mark.gpu


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def _run(name, pairs, n_ret, n_bulk, h_tol, every=(16, 16)):
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
    n = w.N
    # every window row of every (b, h), as the step stored it, within one
    # unit in the last place of the oracle's rotation; far rows (far_offset
    # 0) are the stored keys themselves
    win = np.arange(n - w.W, n)
    kt_win = f64(step.k_tilde[:, :, n - w.W:])
    rng = np.random.default_rng(7)
    for b in range(w.B):
        for h in range(w.H):
            want = oracle.windowed_rope(k[b, h, win], win, n - 1, w.W, w.far_offset, w.rope_base)
            assert_storage_close(kt_win[b, h], want, synth.DTYPES[w.dtype])
    far = np.sort(rng.choice(n - w.W, 512, replace=False))
    assert torch.equal(step.k_tilde[:, :, far].cpu(), k[:, :, far])
    # every (b, h): the whole retrieval split, and the codes of a few
    # retrieval and bulk rows (H and L of the head as the sampled pairs below
    # check them against the oracle)
    Lh = {}
    for h in range(w.H):
        hm = (oracle.query_second_moment(Q[h], w.ridge).astype(np.float32).astype(np.float64)
              if Q is not None else f64(Hg[h]))
        Lo, info = oracle.cholesky(hm)
        assert info == 0
        Lh[h] = Lo.astype(np.float32).astype(np.float64)
    n_r, n_b = every
    for b in range(w.B):
        for h in range(w.H):
            v = oracle.windowed_rope(k[b, h], np.arange(n), n - 1, w.W, w.far_offset, w.rope_base)
            _, cnt, scores, kth = oracle.select_retrieval_set(v, v[-1], w.fraction)
            check_split(perm[b, h], int(count[b, h]), n, cnt, scores, kth)
            ret, bulk = perm[b, h, :cnt], perm[b, h, cnt:n]
            ret = np.sort(rng.choice(ret, min(n_r, len(ret)), replace=False))
            bulk = np.sort(rng.choice(bulk, min(n_b, len(bulk)), replace=False))
            code, d1, d2 = oracle.assign_cholesky(v[ret], c[h], Lh[h])
            check_codes(codes[b, h, ret], code, (d2 - d1) / d2, "retrieval codes")
            code, d1, d2 = oracle.assign_cholesky(v[bulk], c[h], None)
            check_codes(codes[b, h, bulk], code, (d2 - d1) / d2, "bulk codes")
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


@pytest.mark.parametrize("name,b,h", [("llama3_8b_long", 3, 7), ("wide_head", 0, 29)])
def test_rotation_at_the_highest_positions(name, b, h):
    """One whole (sequence, head) of the workload with the window as long as
    the sequence, so every row is rotated at its own position, fp32 out:
    rows near the top position (131071 or 65535), near 2^16 and 2^15, and
    random rows within 2e-6 of the row maximum (the contract is 1e-3)."""
    w = synth.WORKLOADS[name]
    k = synth.head_keys(w, b, h)
    n = w.N
    out = q.a2ats_windowed_rope(dev(k), window=n, far_offset=0, rope_base=w.rope_base,
                                out_dtype=torch.float32)
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([np.arange(n - 256, n), np.arange(65536 - 64, 65536 + 64),
                                     np.arange(32768 - 32, 32768 + 32),
                                     rng.choice(n, 512, replace=False)]))
    rows = rows[rows < n]
    want = oracle.windowed_rope(f64(k[0, 0, rows]), rows, n - 1, n, 0, w.rope_base)
    worst = assert_rows_close(f64(out[0, 0, rows]), want)
    assert worst < 2e-6
