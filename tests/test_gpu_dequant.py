"""GPU parity of a2ats_dequantize against the oracle (v0.39.0 page, "How it
works", step 3: each key reconstructed from its assigned centroid): a
gather, so bit-exact, rows past len untouched, zeros for out-of-range
codes."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import dev, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    # B, H, N, d, dtype, K
    (2, 3, 1000, 128, "bf16", 256),
    (1, 2, 333, 64, "f16", 77),
    (1, 1, 50, 256, "f32", 8),
    (3, 2, 129, 8, "bf16", 5),
])
def test_dequantize_matches_oracle(case):
    B, H, N, d, dt, K = case
    c = synth.gaussian((H, K, d), seed=K + d, dtype=dt)
    rng = np.random.default_rng(N)
    codes = rng.integers(0, K, (B, H, N)).astype(np.int32)
    codes[0, 0, :3] = [-1, K, K + 100]
    lens = torch.tensor([max(N - 31 * b, 1) for b in range(B)], dtype=torch.int32)
    out = torch.full((B, H, N, d), 7.0, dtype=synth.DTYPES[dt], device="cuda")
    q.a2ats_dequantize(dev(torch.from_numpy(codes)), dev(c), lengths=dev(lens), out=out)
    torch.cuda.synchronize()
    got = f64(out.cpu())
    for b in range(B):
        n = int(lens[b])
        for h in range(H):
            want = oracle.dequantize(codes[b, h, :n], f64(c[h]))
            np.testing.assert_array_equal(got[b, h, :n], want)
            assert (got[b, h, n:] == 7.0).all()


def test_dequantize_the_step_codes_full_size():
    """The codes the one-call step writes for the Llama-3.2-3B layer, turned
    back into centroids: each reconstructed row is the centroid the oracle's
    plain VQ picks, on sampled rows (near-ties exempt)."""
    from _parity import check_codes
    w = synth.WORKLOADS["llama32_3b_layer"]
    k, c = synth.keys(w), synth.codebook(w)
    rope = dict(window=w.W, rope_base=w.rope_base)
    _, _, _, codes = q.a2ats_rope_split_plain_assign(dev(k), dev(c), None, w.fraction,
                                                    rope=rope)
    rec = q.a2ats_dequantize(codes, dev(c))
    torch.cuda.synchronize()
    codes, rec = codes.cpu().numpy(), f64(rec.cpu())
    rng = np.random.default_rng(0)
    for h in range(w.H):
        rows = np.sort(rng.choice(w.N - w.W, 256, replace=False))
        np.testing.assert_array_equal(rec[0, h, rows], f64(c[h])[codes[0, h, rows]])
        code, d1, d2 = oracle.assign_cholesky(f64(k[0, h, rows]), f64(c[h]), None)
        check_codes(codes[0, h, rows], code, (d2 - d1) / d2, "codes")
