"""GPU parity of a2ats_code_attention_topk against the oracle: the attention
score of the decode query with every cached key, far keys through their
codes with the far relative position b on the query (deploy-preview
"A2ATS-adapted" page, "Windowed RoPE (Eq. 11-12)": u_ij = q_i R_b k_j^T),
window keys with exact RoPE, and the top tokens by it.  Scores within fp32
rounding of the oracle's fp64 values; the retrieved set exact except for
rows within 1e-5 (of the largest score's magnitude) of the threshold."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import dev, f64

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, N, d, dtype, K, window, far_b, fraction, interleaved
    (2, 3, 1000, 128, "bf16", 256, 64, 2048, 0.1, False),
    (1, 2, 777, 64, "f16", 100, 16, 500, 0.2, True),
    (1, 1, 300, 256, "bf16", 512, 0, 2048, 0.05, False),     # every key far
    (1, 2, 50, 128, "f32", 8, 100, 2048, 0.3, False),        # every key near
    (1, 1, 4099, 128, "bf16", 1024, 512, 4096, 0.02, False),
    (16, 8, 300, 64, "bf16", 64, 32, 1024, 0.1, False),      # many (b, h)
]


def _check(gpu_scores, perm, count, n, want_scores, want_count):
    s = np.asarray(want_scores)
    scale = max(np.abs(s).max(), 1e-30)
    np.testing.assert_allclose(gpu_scores[:n], s, rtol=0, atol=1e-5 * scale)
    assert count == want_count
    p = np.asarray(perm)[:n]
    assert sorted(p.tolist()) == list(range(n))
    ret, bulk = p[:count], p[count:]
    assert (np.diff(ret) > 0).all() and (np.diff(bulk) > 0).all()
    if count:
        kth = np.sort(s)[::-1][count - 1]
        tie = 1e-5 * scale
        inset = np.zeros(n, bool)
        inset[ret] = True
        assert inset[s > kth + tie].all()
        assert not inset[s < kth - tie].any()


@pytest.mark.parametrize("case", CASES)
def test_code_attention_matches_oracle(case):
    B, H, N, d, dt, K, W, b, f, il = case
    k = synth.gaussian((B, H, N, d), seed=N + d, dtype=dt)
    c = synth.gaussian((H, K, d), seed=K + 3, dtype=dt)
    qv = synth.gaussian((B, H, d), seed=N + 11, dtype=dt)
    rng = np.random.default_rng(N)
    codes = rng.integers(0, K, (B, H, N)).astype(np.int32)
    codes[0, 0, :3] = [-1, K, K + 7]  # out of range: score 0
    lens = torch.tensor([max(N - 29 * bb, 1) for bb in range(B)], dtype=torch.int32)
    rope = dict(window=W, rope_base=500000.0, interleaved=int(il))
    scores, perm, count = q.a2ats_code_attention_topk(
        dev(k), dev(torch.from_numpy(codes)), dev(c), dev(qv), f, rope=rope, far_b=b,
        lengths=dev(lens))
    torch.cuda.synchronize()
    scores, perm, count = scores.cpu().numpy(), perm.cpu().numpy(), count.cpu().numpy()
    for bb in range(B):
        n = int(lens[bb])
        for h in range(H):
            _, cnt, s, _ = oracle.code_attention_topk(
                f64(k[bb, h, :n]), n - 1, codes[bb, h, :n], f64(c[h]), f64(qv[bb, h]), W, b,
                500000.0, f, interleaved=il)
            _check(scores[bb, h], perm[bb, h], int(count[bb, h]), n, s, cnt)


def test_code_attention_full_size_sampled():
    """The Llama-3.2-3B layer with the codes of the one-call step: every
    (b, h) scored and ranked against the oracle."""
    w = synth.WORKLOADS["llama32_3b_layer"]
    k, c = synth.keys(w), synth.codebook(w)
    rope = dict(window=w.W, rope_base=w.rope_base)
    kd, cd = dev(k), dev(c)
    _, _, _, codes = q.a2ats_rope_split_plain_assign(kd, cd, None, w.fraction, rope=rope)
    qv = kd[:, :, -1, :].contiguous()  # the newest key as the decode query
    scores, perm, count = q.a2ats_code_attention_topk(kd, codes, cd, qv, 0.02, rope=rope,
                                                      far_b=2048)
    torch.cuda.synchronize()
    scores, perm, count = scores.cpu().numpy(), perm.cpu().numpy(), count.cpu().numpy()
    codes = codes.cpu().numpy()
    for h in range(w.H):
        _, cnt, s, _ = oracle.code_attention_topk(f64(k[0, h]), w.N - 1, codes[0, h], f64(c[h]),
                                                  f64(k[0, h, -1]), w.W, 2048, w.rope_base, 0.02)
        _check(scores[0, h], perm[0, h], int(count[0, h]), w.N, s, cnt)
