"""GPU parity of the sub-vector (product) VQ step, composed from the
assignment calls (dedicated=False), against the oracle's
composition of the same steps (v0.39.0 page, configuration a2ats_sub_dim and
a2ats_codebook_bits, "How it works" steps 1-5; the API page's functions on
[N, sub_dim] sub-vectors): windowed RoPE of the whole head, the split over
tokens, plain VQ of every sub-vector, the H-weighted rule with the
sub_dim x sub_dim factor on the retrieval tokens' sub-vectors, values by
plain VQ."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import check_codes, check_split, dev, f64
from query_aware_vq_gb300.pipeline import A2ATSSubvectorStep

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    # B, H, N, d, sub_dim, K, window, fraction
    (1, 2, 600, 64, 8, 64, 64, 0.1),
    (2, 1, 333, 128, 16, 32, 40, 0.2),
])
def test_subvector_step_matches_oracle(case):
    B, H, N, d, s, K, W, f = case
    G, base = d // s, 500000.0
    k = synth.gaussian((B, H, N, d), seed=N + 1, dtype="bf16")
    v = synth.gaussian((B, H, N, d), seed=N + 2, dtype="f32")
    ck = synth.gaussian((H, K, s), seed=K + 3, dtype="f32")
    cv = synth.gaussian((H, K, s), seed=K + 4, dtype="f32")
    Q = synth.gaussian((H, 4 * N, s), seed=N + 5, dtype="f32")
    Hm = q.a2ats_query_second_moment(dev(Q), 1e-4)
    L, info = q.a2ats_cholesky_factor(Hm)
    lens = torch.tensor([max(N - 41 * b, 1) for b in range(B)], dtype=torch.int32)
    step = A2ATSSubvectorStep(B, H, N, d, s, K, torch.bfloat16, window=W, fraction=f,
                              rope_base=base, dedicated=False)
    step(dev(k), dev(v), dev(ck), dev(cv), L, lengths=dev(lens))
    torch.cuda.synchronize()
    codes_k, codes_v = step.codes_k.cpu().numpy(), step.codes_v.cpu().numpy()
    perm, count = step.perm.cpu().numpy(), step.count.cpu().numpy()
    for h in range(H):
        hm = oracle.query_second_moment(f64(Q[h]), 1e-4).astype(np.float32).astype(np.float64)
        l, inf = oracle.cholesky(hm)
        assert inf == 0
        l = l.astype(np.float32).astype(np.float64)
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
