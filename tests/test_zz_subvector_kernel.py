"""GPU parity of the sub-vector assignment kernel (a2ats_subvector_assign)
against the oracle (v0.39.0 page, configuration a2ats_sub_dim and
a2ats_codebook_bits, "How it works" steps 2 and 5; API page,
a2ats_h_weighted_assignment on sub_dim-wide sub-vectors): every token's
d / sub_dim sub-vectors coded by the per-head table, the H-weighted rule on
the retrieval tokens of a split, plain VQ on the rest and on the values.

The file name sorts last so a stop-at-first-failure run has run every other
test first.
"""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import check_codes, check_split, dev, f64
from query_aware_vq_gb300.pipeline import A2ATSSubvectorStep

pytestmark = pytest.mark.gpu


def _factor(H, s, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(H):
        A = rng.standard_normal((s, s))
        out.append(oracle.cholesky(A @ A.T / s + 0.1 * np.eye(s))[0])
    return np.stack(out).astype(np.float32)


def _split(n, N, frac, rng):
    """A token split in the layout a2ats_select_retrieval_set writes:
    the retrieval tokens ascending, then the bulk ascending."""
    ret = np.sort(rng.choice(n, size=int(np.ceil(frac * n)), replace=False))
    bulk = np.setdiff1d(np.arange(n), ret)
    perm = np.full(N, -7, np.int32)
    perm[:n] = np.concatenate([ret, bulk])
    return perm, len(ret)


@pytest.mark.parametrize("case", [
    # B, H, N, d, sub_dim, K, dtype, rule
    (2, 2, 300, 128, 8, 256, "f32", "split"),
    (1, 3, 200, 64, 16, 64, "bf16", "split"),
    (1, 1, 129, 32, 8, 1024, "f16", "all_weighted"),
    (2, 1, 77, 128, 8, 5, "f32", "plain"),
    (1, 2, 500, 256, 16, 512, "f32", "split"),
])
def test_subvector_assign_matches_oracle(case):
    B, H, N, d, s, K, dt, rule = case
    G = d // s
    x = synth.gaussian((B, H, N, d), seed=N + d, dtype=dt)
    c = synth.gaussian((H, K, s), seed=K + s, dtype=dt)
    L = _factor(H, s, seed=s + K) if rule != "plain" else None
    lens = np.array([max(N - 37 * b, 1) for b in range(B)], np.int32)
    rng = np.random.default_rng(N)
    perm = np.zeros((B, H, N), np.int32)
    count = np.zeros((B, H), np.int32)
    for b in range(B):
        for h in range(H):
            perm[b, h], count[b, h] = _split(int(lens[b]), N, 0.2, rng)
    codes = torch.full((B, H, N, G), -5, dtype=torch.int32, device="cuda")
    split = rule == "split"
    q.a2ats_subvector_assign(
        dev(x), dev(c), s, dev(torch.from_numpy(L)) if L is not None else None,
        lengths=dev(torch.from_numpy(lens)),
        perm=dev(torch.from_numpy(perm)) if split else None,
        count=dev(torch.from_numpy(count)) if split else None, codes=codes)
    torch.cuda.synchronize()
    got = codes.cpu().numpy()
    for b in range(B):
        n = int(lens[b])
        assert (got[b, :, n:] == -5).all()
        for h in range(H):
            sub = f64(x[b, h, :n]).reshape(n * G, s)
            ch = f64(c[h])
            if rule == "plain":
                code, d1, d2 = oracle.assign_cholesky(sub, ch, None)
            elif rule == "all_weighted":
                code, d1, d2 = oracle.assign_cholesky(sub, ch, L[h].astype(np.float64))
            else:
                code, d1, d2 = oracle.assign_cholesky(sub, ch, None)
                ret = perm[b, h, :count[b, h]]
                rsub = (ret[:, None] * G + np.arange(G)).ravel()
                cr, r1, r2 = oracle.assign_cholesky(sub[rsub], ch, L[h].astype(np.float64))
                code[rsub], d1[rsub], d2[rsub] = cr, r1, r2
            check_codes(got[b, h, :n].ravel(), code, (d2 - d1) / np.maximum(d2, 1e-300))


@pytest.mark.parametrize("case", [
    # B, H, N, d, sub_dim, K, window, fraction
    (1, 2, 600, 64, 8, 64, 64, 0.1),
    (2, 1, 333, 128, 16, 32, 40, 0.2),
])
def test_subvector_step_with_the_kernel_matches_oracle(case):
    B, H, N, d, s, K, W, f = case
    G, base = d // s, 500000.0
    k = synth.gaussian((B, H, N, d), seed=N + 1, dtype="bf16")
    v = synth.gaussian((B, H, N, d), seed=N + 2, dtype="f32")
    ck = synth.gaussian((H, K, s), seed=K + 3, dtype="f32")
    cv = synth.gaussian((H, K, s), seed=K + 4, dtype="f32")
    L = torch.from_numpy(_factor(H, s, seed=N))
    lens = torch.tensor([max(N - 41 * b, 1) for b in range(B)], dtype=torch.int32)
    step = A2ATSSubvectorStep(B, H, N, d, s, K, torch.bfloat16, window=W, fraction=f,
                              rope_base=base, dedicated=True)
    step(dev(k), dev(v), dev(ck), dev(cv), dev(L), lengths=dev(lens))
    torch.cuda.synchronize()
    codes_k, codes_v = step.codes_k.cpu().numpy(), step.codes_v.cpu().numpy()
    perm, count = step.perm.cpu().numpy(), step.count.cpu().numpy()
    for h in range(H):
        l = L[h].numpy().astype(np.float64)
        for b in range(B):
            n = int(lens[b])
            kt = oracle.windowed_rope(f64(k[b, h, :n]), np.arange(n), n - 1, W, 0, base)
            _, cnt, scores, kth = oracle.select_retrieval_set(kt, kt[n - 1], f)
            check_split(perm[b, h], int(count[b, h]), n, cnt, scores, kth)
            # the rule each token took is the one its side of the split
            # (checked above) gives it
            ret = np.sort(perm[b, h, :int(count[b, h])])
            sub = kt.reshape(n * G, s)
            code, d1, d2 = oracle.assign_cholesky(sub, f64(ck[h]), None)
            rsub = (ret[:, None] * G + np.arange(G)).ravel()
            code_r, r1, r2 = oracle.assign_cholesky(sub[rsub], f64(ck[h]), l)
            code[rsub], d1[rsub], d2[rsub] = code_r, r1, r2
            check_codes(codes_k[b, h, :n].ravel(), code, (d2 - d1) / d2, "key sub-codes")
            vc, e1, e2 = oracle.assign_cholesky(f64(v[b, h, :n]).reshape(n * G, s), f64(cv[h]),
                                                None)
            check_codes(codes_v[b, h, :n].ravel(), vc, (e2 - e1) / e2, "value sub-codes")


def _blend_expected(sub, c, qfull, beta, rows, G, s):
    """Oracle codes and gaps of the sub-vectors: plain VQ everywhere, then
    the blend with the query's slice g on the sub-vector rows `rows`."""
    code, d1, d2 = oracle.assign_cholesky(sub, c, None)
    gap = (d2 - d1) / np.maximum(d2, 1e-300)
    if beta < 1.0 and len(rows):
        n = sub.shape[0] // G
        qrows = np.tile(qfull.reshape(G, s), (n, 1))
        cb, s1, s2 = oracle.assign_blend(sub[rows], c, qrows[rows], beta)
        code[rows], gap[rows] = cb, s1 - s2
    return code, gap


@pytest.mark.parametrize("case", [
    # B, H, N, d, sub_dim, K, dtype, beta, query, split
    (2, 2, 300, 128, 8, 256, "f32", 0.5, "proxy", True),
    (1, 3, 200, 64, 16, 64, "bf16", 0.0, "given", True),
    (1, 1, 129, 32, 8, 1024, "f16", 0.7, "given", False),
    (2, 1, 77, 128, 8, 5, "f32", 1.0, "proxy", True),
])
def test_subvector_blend_matches_oracle(case):
    B, H, N, d, s, K, dt, beta, qmode, split = case
    G = d // s
    x = synth.gaussian((B, H, N, d), seed=N + 2 * d, dtype=dt)
    c = synth.gaussian((H, K, s), seed=K + 2 * s, dtype=dt)
    qg = synth.gaussian((B, H, d), seed=N + 9, dtype=dt)
    lens = np.array([max(N - 29 * b, 1) for b in range(B)], np.int32)
    rng = np.random.default_rng(N + 1)
    perm = np.zeros((B, H, N), np.int32)
    count = np.zeros((B, H), np.int32)
    for b in range(B):
        for h in range(H):
            perm[b, h], count[b, h] = _split(int(lens[b]), N, 0.25, rng)
    codes = torch.full((B, H, N, G), -5, dtype=torch.int32, device="cuda")
    q.a2ats_subvector_query_aware_assign(
        dev(x), dev(c), s, dev(qg) if qmode == "given" else None, beta,
        lengths=dev(torch.from_numpy(lens)),
        perm=dev(torch.from_numpy(perm)) if split else None,
        count=dev(torch.from_numpy(count)) if split else None, codes=codes)
    torch.cuda.synchronize()
    got = codes.cpu().numpy()
    for b in range(B):
        n = int(lens[b])
        assert (got[b, :, n:] == -5).all()
        for h in range(H):
            sub = f64(x[b, h, :n]).reshape(n * G, s)
            qfull = f64(qg[b, h]) if qmode == "given" else f64(x[b, h, n - 1])
            toks = perm[b, h, :count[b, h]] if split else np.arange(n)
            rows = (np.sort(toks)[:, None] * G + np.arange(G)).ravel()
            code, gap = _blend_expected(sub, f64(c[h]), qfull, beta, rows, G, s)
            check_codes(got[b, h, :n].ravel(), code, gap)


def test_subvector_step_without_a_factor_takes_the_blend():
    """No calibrated H: the step gives the retrieval tokens' sub-vectors the
    cosine blend against the proxy query k~_t, slice by slice."""
    B, H, N, d, s, K, W, f, beta = 1, 2, 500, 64, 8, 64, 64, 0.15, 0.5
    G, base = d // s, 500000.0
    k = synth.gaussian((B, H, N, d), seed=N + 11, dtype="bf16")
    v = synth.gaussian((B, H, N, d), seed=N + 12, dtype="f32")
    ck = synth.gaussian((H, K, s), seed=K + 13, dtype="f32")
    cv = synth.gaussian((H, K, s), seed=K + 14, dtype="f32")
    step = A2ATSSubvectorStep(B, H, N, d, s, K, torch.bfloat16, window=W, fraction=f,
                              rope_base=base, beta=beta)
    step(dev(k), dev(v), dev(ck), dev(cv), None)
    torch.cuda.synchronize()
    codes_k, codes_v = step.codes_k.cpu().numpy(), step.codes_v.cpu().numpy()
    perm, count = step.perm.cpu().numpy(), step.count.cpu().numpy()
    for h in range(H):
        n = N
        kt = oracle.windowed_rope(f64(k[0, h]), np.arange(n), n - 1, W, 0, base)
        _, cnt, scores, kth = oracle.select_retrieval_set(kt, kt[n - 1], f)
        check_split(perm[0, h], int(count[0, h]), n, cnt, scores, kth)
        ret = np.sort(perm[0, h, :int(count[0, h])])
        rows = (ret[:, None] * G + np.arange(G)).ravel()
        code, gap = _blend_expected(kt.reshape(n * G, s), f64(ck[h]), kt[n - 1], beta, rows,
                                    G, s)
        check_codes(codes_k[0, h].ravel(), code, gap, "key sub-codes")
        vc, e1, e2 = oracle.assign_cholesky(f64(v[0, h]).reshape(n * G, s), f64(cv[h]), None)
        check_codes(codes_v[0, h].ravel(), vc, (e2 - e1) / e2, "value sub-codes")


def test_config_without_query_awareness_codes_every_token_plainly():
    """A2ATSConfig(use_query_aware=False): the split is empty and every key
    and value sub-vector takes plain VQ."""
    from query_aware_vq_gb300.config import A2ATSConfig

    cfg = A2ATSConfig(head_dim=64, window=32, use_query_aware=False, rope_base=500000.0)
    B, H, N = 1, 2, 300
    s, G, K = cfg.sub_dim, 64 // cfg.sub_dim, cfg.n_centroids
    k = synth.gaussian((B, H, N, 64), seed=61, dtype="bf16")
    v = synth.gaussian((B, H, N, 64), seed=62, dtype="f32")
    ck = synth.gaussian((H, K, s), seed=63, dtype="f32")
    cv = synth.gaussian((H, K, s), seed=64, dtype="f32")
    step = cfg.subvector_step(B, H, N, torch.bfloat16)
    step(dev(k), dev(v), dev(ck), dev(cv), None)
    torch.cuda.synchronize()
    assert step.count.cpu().numpy().tolist() == [[0] * H]
    for h in range(H):
        kt = oracle.windowed_rope(f64(k[0, h]), np.arange(N), N - 1, cfg.window, 0,
                                  cfg.rope_base)
        code, d1, d2 = oracle.assign_cholesky(kt.reshape(N * G, s), f64(ck[h]), None)
        check_codes(step.codes_k[0, h].cpu().numpy().ravel(), code, (d2 - d1) / d2)
        vc, e1, e2 = oracle.assign_cholesky(f64(v[0, h]).reshape(N * G, s), f64(cv[h]), None)
        check_codes(step.codes_v[0, h].cpu().numpy().ravel(), vc, (e2 - e1) / e2)


def test_config_factor_drives_the_h_weighted_rule():
    """A2ATSConfig.factor: L of a shared query_h for every head; the step
    with it gives the retrieval tokens' sub-vectors the H-weighted rule."""
    from query_aware_vq_gb300.config import A2ATSConfig

    rng = np.random.default_rng(71)
    A = rng.standard_normal((8, 8))
    hq = A @ A.T / 8 + 0.1 * np.eye(8)
    cfg = A2ATSConfig(head_dim=64, window=32, query_h=hq, retrieval_fraction=0.2,
                      rope_base=500000.0)
    B, H, N = 1, 2, 300
    s, G, K = cfg.sub_dim, 64 // cfg.sub_dim, cfg.n_centroids
    L = cfg.factor(H)
    lo, _ = oracle.cholesky(hq.astype(np.float32).astype(np.float64))
    for h in range(H):
        np.testing.assert_allclose(f64(L[h]), lo, rtol=0, atol=1e-5)
    k = synth.gaussian((B, H, N, 64), seed=72, dtype="bf16")
    v = synth.gaussian((B, H, N, 64), seed=73, dtype="f32")
    ck = synth.gaussian((H, K, s), seed=74, dtype="f32")
    cv = synth.gaussian((H, K, s), seed=75, dtype="f32")
    step = cfg.subvector_step(B, H, N, torch.bfloat16)
    step(dev(k), dev(v), dev(ck), dev(cv), L)
    torch.cuda.synchronize()
    perm, count = step.perm.cpu().numpy(), step.count.cpu().numpy()
    for h in range(H):
        lh = f64(L[h])
        kt = oracle.windowed_rope(f64(k[0, h]), np.arange(N), N - 1, cfg.window, 0,
                                  cfg.rope_base)
        ret = np.sort(perm[0, h, :int(count[0, h])])
        sub = kt.reshape(N * G, s)
        code, d1, d2 = oracle.assign_cholesky(sub, f64(ck[h]), None)
        rsub = (ret[:, None] * G + np.arange(G)).ravel()
        cr, r1, r2 = oracle.assign_cholesky(sub[rsub], f64(ck[h]), lh)
        code[rsub], d1[rsub], d2[rsub] = cr, r1, r2
        check_codes(step.codes_k[0, h].cpu().numpy().ravel(), code, (d2 - d1) / d2)
