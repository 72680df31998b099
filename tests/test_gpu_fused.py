"""GPU parity of a2ats_rope_split_plain_assign, the one call for the
windowed RoPE (deploy-preview page "A2ATS-adapted", "Per-step re-rotation"),
the retrieval split (API page, a2ats_select_retrieval_set) and the bulk rule
of the v0.39.0 page's routing ("How it works", step 2: the nearest
centroid).  Its k~ and codes equal those of the separate calls bit for bit;
its split is checked against the oracle (exact except on near-ties, whose
scores may differ in the last bits between the fused and separate paths)."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import assert_storage_close, check_split, dev, f64

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, N, d, dtype, K, fraction, rope
    (2, 3, 1000, 128, "bf16", 256, 0.1, dict(window=64, rope_base=500000.0)),
    (2, 1, 300, 128, "bf16", 300, 0.3, dict(window=40, rope_base=10000.0, interleaved=1)),
    (1, 2, 700, 256, "bf16", 512, 0.1, dict(window=0, rope_base=10000.0)),
    (1, 2, 1500, 192, "f16", 1000, 0.05, dict(window=129, rope_base=10000.0)),
    (2, 2, 900, 64, "bf16", 64, 0.2, dict(window=5000, rope_base=500000.0)),  # all in window
    (1, 1, 4099, 128, "f16", 1024, 0.02, dict(window=512, rope_base=500000.0)),
    # no one-pass form: far rows rotated, fp32 keys, widths off the tensor-core path
    (1, 2, 777, 64, "f16", 128, 0.2, dict(window=16, far_offset=5, rope_base=10000.0)),
    (1, 2, 300, 24, "f32", 32, 0.3, dict(window=8, rope_base=10000.0)),
    (1, 1, 5, 16, "bf16", 4, 0.5, dict(window=2, rope_base=10000.0)),
]


def _lens(B, N):
    return dev(torch.tensor([max(N - 37 * b, 1) for b in range(B)], dtype=torch.int32))


@pytest.mark.parametrize("case", CASES)
def test_fused_call_equals_the_separate_calls(case):
    B, H, N, d, dt, K, f, rope = case
    k = synth.gaussian((B, H, N, d), seed=N + 11, dtype=dt)
    c = synth.gaussian((H, K, d), seed=K + 5, dtype=dt)
    kd, cd, lens = dev(k), dev(c), _lens(B, N)
    want_out = torch.zeros((B, H, N, d), dtype=kd.dtype, device="cuda")
    q.a2ats_windowed_rope(kd, lengths=lens, out=want_out, **rope)
    want_codes = q.a2ats_h_weighted_assign(kd, cd, None, lengths=lens, rope=rope, rows="all")
    out = torch.zeros_like(want_out)
    codes = torch.full((B, H, N), -7, dtype=torch.int32, device="cuda")
    out, perm, count, codes = q.a2ats_rope_split_plain_assign(
        kd, cd, None, f, rope=rope, lengths=lens, out=out, codes=codes)
    torch.cuda.synchronize()
    perm, count = perm.cpu().numpy(), count.cpu().numpy()
    for b in range(B):
        n = int(lens[b])
        assert torch.equal(out[b, :, :n], want_out[b, :, :n])
        assert torch.equal(codes[b, :, :n], want_codes[b, :, :n])
        # rows past len are not written
        assert (out[b, :, n:] == 0).all()
        assert (codes[b, :, n:] == -7).all()
        for h in range(H):
            v = oracle.windowed_rope(f64(k[b, h, :n]), np.arange(n), n - 1, rope["window"],
                                     rope.get("far_offset", 0), rope["rope_base"],
                                     interleaved=bool(rope.get("interleaved", 0)))
            _, cnt, scores, kth = oracle.select_retrieval_set(v, v[n - 1], f)
            check_split(perm[b, h], int(count[b, h]), n, cnt, scores, kth)


def test_fused_split_event_and_reuse():
    """split_done orders a second stream after the split; reuse=True on new
    keys gives what a fresh call gives."""
    B, H, N, d, K = 2, 4, 3000, 128, 512
    rope = dict(window=256, rope_base=500000.0)
    c = dev(synth.gaussian((H, K, d), seed=1, dtype="bf16"))
    lens = _lens(B, N)
    lib = q.library()
    ws = torch.empty(lib.a2ats_rope_split_plain_assign_workspace_size(B, H, N, d, K),
                     dtype=torch.uint8, device="cuda")
    ev = torch.cuda.Event()
    ev.record()
    side = torch.cuda.Stream()
    for i, seed in enumerate((2, 3)):
        k = dev(synth.gaussian((B, H, N, d), seed=seed, dtype="bf16"))
        out, perm, count, codes = q.a2ats_rope_split_plain_assign(
            k, c, None, 0.05, rope=rope, lengths=lens, reuse=i > 0, split_done=ev, workspace=ws)
        side.wait_event(ev)
        with torch.cuda.stream(side):
            perm_seen, count_seen = perm.clone(), count.clone()
        torch.cuda.synchronize()
        assert torch.equal(perm_seen, perm) and torch.equal(count_seen, count)
        out2, perm2, count2, codes2 = q.a2ats_rope_split_plain_assign(
            k, c, None, 0.05, rope=rope, lengths=lens)
        torch.cuda.synchronize()
        assert torch.equal(count, count2)
        for b in range(B):
            n = int(lens[b])   # rows past len are not written
            assert torch.equal(codes[b, :, :n], codes2[b, :, :n])
            assert torch.equal(out[b, :, :n], out2[b, :, :n])
            assert torch.equal(perm[b, :, :n], perm2[b, :, :n])


def test_fused_full_size_sampled():
    """The bench's launch: the Llama-3.2-3B layer at full size, codes of
    sampled rows and every (b, h) split against the oracle."""
    w = synth.WORKLOADS["llama32_3b_layer"]
    k, c = synth.keys(w), synth.codebook(w)
    rope = dict(window=w.W, far_offset=w.far_offset, rope_base=w.rope_base)
    out, perm, count, codes = q.a2ats_rope_split_plain_assign(dev(k), dev(c), None, w.fraction,
                                                              rope=rope)
    torch.cuda.synchronize()
    perm, count, codes = perm.cpu().numpy(), count.cpu().numpy(), codes.cpu().numpy()
    kt = out.cpu()
    rng = np.random.default_rng(0)
    from _parity import check_codes
    for b in range(w.B):
        for h in range(w.H):
            v = oracle.windowed_rope(k[b, h], np.arange(w.N), w.N - 1, w.W, 0, w.rope_base)
            _, cnt, scores, kth = oracle.select_retrieval_set(v, v[-1], w.fraction)
            check_split(perm[b, h], int(count[b, h]), w.N, cnt, scores, kth)
            rows = np.unique(np.concatenate([rng.choice(w.N, 512, replace=False),
                                             np.arange(w.N - w.W - 2, w.N)]))
            # far rows are the stored keys themselves; window rows within one
            # unit in the last place of the oracle's rotation
            far = rows[rows < w.N - w.W]
            assert torch.equal(kt[b, h, far], k[b, h, far])
            win = rows[rows >= w.N - w.W]
            assert_storage_close(f64(kt[b, h, win]), v[win], kt.dtype)
            code, d1, d2 = oracle.assign_cholesky(v[rows], c[h], None)
            check_codes(codes[b, h, rows], code, (d2 - d1) / d2, "codes")
