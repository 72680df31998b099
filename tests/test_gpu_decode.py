"""GPU parity of the decode step (v0.39.0 page, "How it works": the incoming
key is stored, the whole cache is re-rotated against the new decode position,
the retrieval split is recomputed over every cached key, and the incoming key
is assigned with itself as the proxy query) against the oracle, step by step,
plus the streaming workload of 64 sequences at its full size (sampled)."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import assert_storage_close, check_codes, check_split, dev, f64
from query_aware_vq_gb300.pipeline import A2ATSDecodeStep

pytestmark = pytest.mark.gpu


def _check_step(step, cache, lengths, codebook, W, base, f, beta, pairs, L=None):
    lens = lengths.cpu().numpy()
    perm, count = step.perm.cpu().numpy(), step.count.cpu().numpy()
    codes = step.codes.cpu().numpy()
    kt = step.k_tilde
    for b, h in pairs:
        n = int(lens[b])
        k = f64(cache[b, h, :n])
        v = oracle.windowed_rope(k, np.arange(n), n - 1, W, 0, base)
        _, cnt, scores, kth = oracle.select_retrieval_set(v, v[-1], f)
        check_split(perm[b, h], int(count[b, h]), n, cnt, scores, kth)
        # the rotated cache at the new position (storage dtype)
        rs = np.arange(max(0, n - W - 2), n)
        assert_storage_close(f64(kt[b, h, rs]), v[rs], kt.dtype)
        # the new key's code
        if L is None:
            code, s1, s2 = oracle.assign_blend(v[-1:], codebook[h], v[-1], beta)
            gap = (s1 - s2) if beta != 1.0 else (s2 - s1) / s2
        else:
            code, d1, d2 = oracle.assign_cholesky(v[-1:], codebook[h], L[h])
            gap = (d2 - d1) / d2
        check_codes(codes[b, h, n - 1:n], code, gap, "new-key code")


@pytest.mark.parametrize("hweighted", [False, True])
def test_decode_steps_match_oracle(hweighted):
    B, H, N, d, K, W, f, beta, base = 3, 2, 700, 128, 64, 32, 0.1, 0.7, 500000.0
    w = synth.scaled(synth.WORKLOADS["decode_stream"], B=B, H=H, N=N, K=K, W=W)
    cache = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
    lens0 = [300, 451, 512]
    full = synth.keys(synth.scaled(w, N=600))
    for b in range(B):
        cache[b, :, :lens0[b]] = full[b, :, :lens0[b]]
    cache = dev(cache)
    lengths = dev(torch.tensor(lens0, dtype=torch.int32))
    cb = synth.codebook(w)
    L = None
    if hweighted:
        rng = np.random.default_rng(3)
        Ls = []
        for _ in range(H):
            g = rng.standard_normal((d, 2 * d))
            Ls.append(oracle.cholesky(g @ g.T / (2 * d) + 1e-2 * np.eye(d))[0])
        L = torch.from_numpy(np.stack(Ls).astype(np.float32))
    step = A2ATSDecodeStep(B, H, N, d, K, torch.bfloat16, window=W, fraction=f, rope_base=base,
                           beta=beta)
    for s in range(3):
        new = dev(synth.decode_new_keys(w, s))
        step(cache, lengths, new, dev(cb), L=dev(L) if L is not None else None)
        torch.cuda.synchronize()
        assert lengths.cpu().tolist() == [x + s + 1 for x in lens0]
        for b in range(B):
            assert torch.equal(cache[b, :, int(lengths[b]) - 1].cpu(), new[b].cpu())
        _check_step(step, cache, lengths, cb, W, base, f, beta,
                    [(b, h) for b in range(B) for h in range(H)], L)


def test_append_leaves_full_sequences_alone():
    cache = dev(torch.zeros((2, 1, 4, 16), dtype=torch.bfloat16))
    lengths = dev(torch.tensor([4, 1], dtype=torch.int32))
    q.a2ats_append_rows(cache, lengths, dev(torch.ones((2, 1, 16), dtype=torch.bfloat16)))
    assert lengths.cpu().tolist() == [4, 2]
    assert (cache[0] == 0).all() and (cache[1, 0, 1] == 1).all()


def test_decode_stream_full_size_sampled():
    w = synth.WORKLOADS["decode_stream"]
    lens0 = synth.decode_lengths(w)
    keys = synth.keys(synth.scaled(w, N=int(lens0.max())))
    cache = torch.zeros((w.B, w.H, w.N, w.d), dtype=torch.bfloat16)
    cache[:, :, :keys.shape[2]] = keys
    del keys
    cache = dev(cache)
    lengths = dev(torch.from_numpy(lens0))
    cb = synth.codebook(w)
    step = A2ATSDecodeStep(w.B, w.H, w.N, w.d, w.K, torch.bfloat16, window=w.W,
                           fraction=w.fraction, rope_base=w.rope_base, beta=w.betas[0])
    rng = np.random.default_rng(0)
    for s in range(2):
        step(cache, lengths, dev(synth.decode_new_keys(w, s)), dev(cb))
        torch.cuda.synchronize()
        pairs = [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(3)]
        _check_step(step, cache, lengths, cb, w.W, w.rope_base, w.fraction, w.betas[0], pairs)
    # every new key's code against the oracle (512 rows)
    lens = lengths.cpu().numpy()
    codes = step.codes.cpu().numpy()
    for b in range(w.B):
        n = int(lens[b])
        for h in range(w.H):
            k = f64(cache[b, h, n - 1:n])
            v = oracle.rope_row(k[0], n - 1, w.rope_base)[None]
            code, s1, s2 = oracle.assign_blend(v, cb[h], v[0], w.betas[0])
            check_codes(codes[b, h, n - 1:n], code, s1 - s2, "new-key code")
