"""GPU parity: H-weighted and cosine-blend assignment against the oracle
(API page, a2ats_h_weighted_assignment and a2ats_query_aware_assignment).
Codes must equal the oracle's except where its top-2 gap is below 1e-5."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import check_codes, dev, f64

pytestmark = pytest.mark.gpu


def _spd(rng, d, cond):
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    lam = np.exp(np.linspace(0, np.log(cond), d))
    return (Qm * lam) @ Qm.T


def _L(H, d, cond, seed):
    rng = np.random.default_rng(seed)
    Ls = []
    for _ in range(H):
        l, _ = oracle.cholesky(_spd(rng, d, cond))
        Ls.append(l)
    return torch.from_numpy(np.stack(Ls).astype(np.float32))


def _rows(x, lens, rope):
    """Per (b, h): the oracle's k~ of the valid rows (fp64)."""
    B, H, N, d = x.shape
    out = {}
    for b in range(B):
        n = int(lens[b])
        for h in range(H):
            v = f64(x[b, h, :n])
            if rope is not None:
                v = oracle.windowed_rope(v, np.arange(n), n - 1, rope["window"],
                                         rope.get("far_offset", 0), rope["rope_base"])
            out[b, h] = v
    return out


CASES = [
    # B, H, N, d, K, dtype, with L, rope
    (2, 2, 300, 128, 100, "bf16", True, None),
    (1, 3, 129, 64, 33, "f32", False, None),
    (2, 1, 200, 128, 64, "f16", True, dict(window=40, far_offset=0, rope_base=500000.0)),
    (1, 2, 150, 256, 40, "bf16", True, dict(window=20, far_offset=9, rope_base=10000.0)),
    (1, 1, 70, 24, 17, "f32", True, None),
    (1, 1, 5, 16, 1, "bf16", False, None),
    # every row inside the window: all rows take the two-plane pass
    (1, 2, 600, 128, 700, "bf16", True, dict(window=10 ** 6, far_offset=0, rope_base=500000.0)),
    # far rows rotated at a fixed offset (rotated codebook) next to exact in-window rows
    (2, 1, 300, 64, 257, "f16", False, dict(window=50, far_offset=3, rope_base=10000.0)),
    (1, 2, 400, 128, 33, "bf16", False, dict(window=128, far_offset=11, rope_base=500000.0)),
    (1, 1, 1000, 256, 513, "f16", True, dict(window=300, far_offset=0, rope_base=10000.0)),
    # more than 2048 centroids: the pass over the stored keys takes one row
    # block per tile and 256-column accumulators
    (2, 1, 700, 128, 2500, "bf16", True, dict(window=64, far_offset=0, rope_base=500000.0)),
    (1, 2, 400, 64, 3000, "f16", False, None),
]


@pytest.mark.parametrize("case", CASES)
def test_h_weighted_matches_oracle(case):
    B, H, N, d, K, dt, withL, rope = case
    x = synth.gaussian((B, H, N, d), seed=N, dtype=dt, scale=2.0)
    c = synth.gaussian((H, K, d), seed=K + 1, dtype=dt, scale=2.0)
    L = _L(H, d, 30.0, seed=d) if withL else None
    lens = torch.tensor([N - 11 * b for b in range(B)], dtype=torch.int32)
    codes = q.a2ats_h_weighted_assign(dev(x), dev(c), dev(L) if withL else None,
                                      lengths=dev(lens), rope=rope)
    got = codes.cpu().numpy()
    kt = _rows(x, lens, rope)
    for (b, h), v in kt.items():
        code, d1, d2 = oracle.assign_cholesky(v, c[h], L[h] if withL else None)
        check_codes(got[b, h, :len(v)], code, (d2 - d1) / np.maximum(d2, 1e-300))


@pytest.mark.parametrize("dt,withL", [("bf16", False), ("bf16", True), ("f16", True),
                                      ("f32", False)])
def test_single_centroid_gives_code_zero(dt, withL):
    """K = 1: the one centroid is every row's nearest (its second distance
    is infinite, so no row is a near tie)."""
    B, H, N, d = 2, 2, 333, 128
    x = synth.gaussian((B, H, N, d), seed=5, dtype=dt, scale=2.0)
    c = synth.gaussian((H, 1, d), seed=6, dtype=dt, scale=2.0)
    L = _L(H, d, 30.0, seed=1) if withL else None
    codes = torch.full((B, H, N), -3, dtype=torch.int32, device="cuda")
    q.a2ats_h_weighted_assign(dev(x), dev(c), dev(L) if withL else None, codes=codes,
                              rope=dict(window=40, far_offset=0, rope_base=10000.0))
    assert (codes.cpu() == 0).all()


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("f32", 48)])
def test_entries_above_the_diagonal_are_ignored(dt, d):
    """Only the lower triangle of L is read: filling the rest with noise
    changes no code, on the tensor-core route and on the SIMT route."""
    B, H, N, K = 1, 2, 300, 70
    x = dev(synth.gaussian((B, H, N, d), seed=31, dtype=dt, scale=2.0))
    c = dev(synth.gaussian((H, K, d), seed=32, dtype=dt, scale=2.0))
    L = _L(H, d, 30.0, seed=33)
    noisy = L + torch.triu(torch.from_numpy(
        np.random.default_rng(34).standard_normal((H, d, d)).astype(np.float32)), diagonal=1)
    rope = dict(window=40, far_offset=0, rope_base=500000.0)
    a = q.a2ats_h_weighted_assign(x, c, dev(L), rope=rope)
    b = q.a2ats_h_weighted_assign(x, c, dev(noisy), rope=rope)
    assert torch.equal(a, b)


@pytest.mark.parametrize("mode", ["retrieval", "bulk"])
@pytest.mark.parametrize("rope", [None, dict(window=40, far_offset=5, rope_base=10000.0)])
def test_row_selection_writes_only_its_rows(mode, rope):
    B, H, N, d, K = 1, 2, 300, 128, 50
    x = synth.gaussian((B, H, N, d), seed=7, dtype="bf16")
    c = synth.gaussian((H, K, d), seed=8, dtype="bf16")
    perm = np.zeros((B, H, N), np.int32)
    count = np.zeros((B, H), np.int32)
    for h in range(H):
        p, cnt, _, _ = oracle.select_retrieval_set(x[0, h], f64(x[0, h, -1]), 0.2)
        perm[0, h], count[0, h] = p, cnt
    codes = torch.full((B, H, N), -7, dtype=torch.int32, device="cuda")
    q.a2ats_h_weighted_assign(dev(x), dev(c), None, rope=rope, rows=mode,
                              perm=dev(torch.from_numpy(perm)),
                              count=dev(torch.from_numpy(count)), codes=codes)
    got = codes.cpu().numpy()
    kt = _rows(x, torch.tensor([N], dtype=torch.int32), rope)
    for h in range(H):
        sel = perm[0, h, :count[0, h]] if mode == "retrieval" else perm[0, h, count[0, h]:]
        other = np.setdiff1d(np.arange(N), sel)
        assert (got[0, h, other] == -7).all()
        code, d1, d2 = oracle.assign_cholesky(kt[0, h][sel], c[h], None)
        check_codes(got[0, h, sel], code, (d2 - d1) / d2)


@pytest.mark.parametrize("beta", [0.0, 0.3, 0.7, 1.0])
@pytest.mark.parametrize("qmode", ["given", "proxy"])
def test_blend_matches_oracle(beta, qmode):
    B, H, N, d, K = 2, 2, 260, 128, 90
    x = synth.gaussian((B, H, N, d), seed=11, dtype="bf16", scale=2.0)
    c = synth.gaussian((H, K, d), seed=12, dtype="bf16", scale=2.0)
    lens = torch.tensor([N, N - 40], dtype=torch.int32)
    rope = dict(window=32, far_offset=0, rope_base=500000.0)
    query = synth.gaussian((B, H, d), seed=13, dtype="bf16") if qmode == "given" else None
    codes = q.a2ats_query_aware_assign(dev(x), dev(c), dev(query) if query is not None else None,
                                       beta, lengths=dev(lens), rope=rope)
    got = codes.cpu().numpy()
    kt = _rows(x, lens, rope)
    for (b, h), v in kt.items():
        qv = f64(query[b, h]) if query is not None else v[-1]
        code, s1, s2 = oracle.assign_blend(v, c[h], qv, beta)
        gap = (s2 - s1) / np.maximum(s2, 1e-300) if beta == 1.0 else (s1 - s2)
        check_codes(got[b, h, :len(v)], code, gap)


def test_beta_one_equals_plain_vq_bitwise():
    x = dev(synth.gaussian((1, 2, 300, 128), seed=21, dtype="bf16"))
    c = dev(synth.gaussian((2, 64, 128), seed=22, dtype="bf16"))
    a = q.a2ats_query_aware_assign(x, c, None, 1.0)
    b = q.a2ats_h_weighted_assign(x, c, None)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["llama32_3b_layer"])
def test_h_weighted_full_size_sampled(name):
    w = synth.WORKLOADS[name]
    k, c = synth.keys(w), synth.codebook(w)
    Q = synth.queries(w)
    Ls = []
    for h in range(w.H):
        hm = oracle.query_second_moment(Q[h], w.ridge).astype(np.float32)
        Ls.append(oracle.cholesky(hm.astype(np.float64))[0].astype(np.float32))
    L = torch.from_numpy(np.stack(Ls))
    rope = dict(window=w.W, far_offset=w.far_offset, rope_base=w.rope_base)
    got = q.a2ats_h_weighted_assign(dev(k), dev(c), dev(L), rope=rope).cpu().numpy()
    rng = np.random.default_rng(1)
    for h in range(w.H):
        rows = np.unique(np.concatenate([rng.choice(w.N, 512, replace=False),
                                         np.arange(w.N - 64, w.N)]))
        v = oracle.windowed_rope(k[0, h, rows], rows, w.N - 1, w.W, 0, w.rope_base)
        code, d1, d2 = oracle.assign_cholesky(v, c[h], L[h])
        check_codes(got[0, h, rows], code, (d2 - d1) / d2)


@pytest.mark.parametrize("dt,d,withL,rows,rope", [
    ("bf16", 128, True, "retrieval", dict(window=40, far_offset=0, rope_base=500000.0)),
    ("bf16", 128, False, "bulk", dict(window=40, far_offset=0, rope_base=500000.0)),
    ("f16", 64, True, "all", dict(window=30, far_offset=3, rope_base=10000.0)),
    ("f32", 48, True, "retrieval", None),   # the SIMT route
])
def test_reuse_takes_the_codebook_side_from_the_workspace(dt, d, withL, rows, rope):
    """A call with reuse gives, on new keys, the codes a full call gives."""
    B, H, N, K = 2, 2, 400, 90
    c = dev(synth.gaussian((H, K, d), seed=41, dtype=dt, scale=2.0))
    L = dev(_L(H, d, 30.0, seed=42)) if withL else None
    lens = dev(torch.tensor([N, N - 33], dtype=torch.int32))
    perm = count = None
    lib = q.library()
    ws = torch.empty(lib.a2ats_h_weighted_assign_workspace_size(B, H, N, d, K), dtype=torch.uint8,
                     device="cuda")
    for step, seed in enumerate((43, 44, 45)):
        x = dev(synth.gaussian((B, H, N, d), seed=seed, dtype=dt, scale=2.0))
        if rows in ("retrieval", "bulk"):
            perm, count = q.a2ats_select_retrieval_set(x, None, 0.1, lengths=lens, rope=rope)
        kw = dict(lengths=lens, rope=rope, rows=rows, perm=perm, count=count)
        want = q.a2ats_h_weighted_assign(x, c, L, **kw)
        got = torch.full_like(want, -5)
        got = q.a2ats_h_weighted_assign(x, c, L, codes=got, workspace=ws, reuse=step > 0, **kw)
        torch.cuda.synchronize()
        if rows == "all":
            for b in range(B):
                n = int(lens[b])
                assert torch.equal(got[b, :, :n], want[b, :, :n])
        else:
            for b in range(B):
                for h in range(H):
                    n, cnt = int(lens[b]), int(count[b, h])
                    sel = perm[b, h, :cnt] if rows == "retrieval" else perm[b, h, cnt:n]
                    assert torch.equal(got[b, h, sel.long()], want[b, h, sel.long()])


@pytest.mark.parametrize("dt,d,beta,rows,rope", [
    ("bf16", 128, 0.7, "last", dict(window=40, far_offset=0, rope_base=500000.0)),
    ("bf16", 128, 0.7, "all", dict(window=40, far_offset=0, rope_base=500000.0)),
    ("bf16", 128, 1.0, "all", dict(window=40, far_offset=0, rope_base=500000.0)),  # tensor cores
    ("f32", 48, 0.5, "all", None),
])
def test_blend_reuse_takes_the_codebook_side_from_the_workspace(dt, d, beta, rows, rope):
    """The cosine blend with reuse gives, on new keys, the codes a full call
    gives (the decoded centroids and norms, or for beta = 1 the planes, come
    from the workspace)."""
    B, H, N, K = 2, 2, 400, 90
    c = dev(synth.gaussian((H, K, d), seed=51, dtype=dt, scale=2.0))
    lens = dev(torch.tensor([N, N - 33], dtype=torch.int32))
    lib = q.library()
    ws = torch.empty(lib.a2ats_query_aware_assign_workspace_size(B, H, N, d, K),
                     dtype=torch.uint8, device="cuda")
    for step, seed in enumerate((53, 54, 55)):
        x = dev(synth.gaussian((B, H, N, d), seed=seed, dtype=dt, scale=2.0))
        kw = dict(lengths=lens, rope=rope, rows=rows)
        want = q.a2ats_query_aware_assign(x, c, None, beta, **kw)
        got = torch.full_like(want, -5)
        got = q.a2ats_query_aware_assign(x, c, None, beta, codes=got, workspace=ws,
                                         reuse=step > 0, **kw)
        torch.cuda.synchronize()
        for b in range(B):
            n = int(lens[b])
            if rows == "last":
                assert torch.equal(got[b, :, n - 1], want[b, :, n - 1])
            else:
                assert torch.equal(got[b, :, :n], want[b, :, :n])
