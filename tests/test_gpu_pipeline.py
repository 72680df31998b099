"""GPU parity of one whole step (calibration -> windowed RoPE -> retrieval
split -> routed assignment) against the oracle's composition of the same
steps (v0.39.0 page, "How it works"; deploy-preview page, "Per-step
re-rotation").  H and L are float32 arrays on the API page, so the oracle's
own H and L are rounded to fp32 where the pages' functions return them."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import assert_storage_close, check_codes, check_split, dev, f64
from query_aware_vq_gb300.pipeline import A2ATSStep

pytestmark = pytest.mark.gpu


def _oracle_L(Q, ridge):
    hm = oracle.query_second_moment(Q, ridge).astype(np.float32).astype(np.float64)
    l, info = oracle.cholesky(hm)
    assert info == 0
    return l.astype(np.float32).astype(np.float64)


def _run(w, rows_sample=None, beta_path=False, seed=0, fused=True):
    k, c = synth.keys(w), synth.codebook(w)
    Q = None if beta_path else synth.queries(w)
    step = A2ATSStep(w.B, w.H, w.N, w.d, w.K, synth.DTYPES[w.dtype], window=w.W,
                     fraction=w.fraction, rope_base=w.rope_base, far_offset=w.far_offset,
                     M=w.M, ridge=w.ridge, beta=w.betas[-1], fused=fused)
    kd, cd = dev(k), dev(c)
    step(kd, cd, queries=dev(Q) if Q is not None else None)
    torch.cuda.synchronize()
    codes, perm, count = step.codes.cpu().numpy(), step.perm.cpu().numpy(), step.count.cpu().numpy()
    kt = f64(step.k_tilde)
    rng = np.random.default_rng(seed)
    for b in range(w.B):
        for h in range(w.H):
            n = w.N
            L = None if beta_path else _oracle_L(f64(Q[h]), w.ridge)
            v = oracle.windowed_rope(k[b, h], np.arange(n), n - 1, w.W, w.far_offset, w.rope_base)
            _, cnt, scores, kth = oracle.select_retrieval_set(v, v[-1], w.fraction)
            check_split(perm[b, h], int(count[b, h]), n, cnt, scores, kth)
            # the written k~ (storage dtype) against the oracle, sampled rows
            rs = np.unique(np.concatenate([rng.choice(n, min(n, 256), replace=False),
                                           np.arange(max(0, n - w.W - 1), n)]))
            assert_storage_close(kt[b, h, rs], v[rs], synth.DTYPES[w.dtype])
            ret = perm[b, h, :cnt]
            bulk = perm[b, h, cnt:]
            if rows_sample is not None and len(bulk) > rows_sample:
                bulk = np.sort(rng.choice(bulk, rows_sample, replace=False))
            if len(ret):
                if beta_path:
                    code, s1, s2 = oracle.assign_blend(v[ret], c[h], v[-1], w.betas[-1])
                    gap = (s2 - s1) / s2 if w.betas[-1] == 1.0 else s1 - s2
                else:
                    code, d1, d2 = oracle.assign_cholesky(v[ret], c[h], L)
                    gap = (d2 - d1) / d2
                check_codes(codes[b, h, ret], code, gap, "retrieval codes")
            code, d1, d2 = oracle.assign_cholesky(v[bulk], c[h], None)
            check_codes(codes[b, h, bulk], code, (d2 - d1) / d2, "bulk codes")
    return step


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("beta_path", [False, True])
def test_step_tiny(beta_path, fused):
    _run(synth.WORKLOADS["tiny"], beta_path=beta_path, fused=fused)


@pytest.mark.parametrize("fused", [True, False])
def test_step_llama32_3b_layer_sampled(fused):
    _run(synth.WORKLOADS["llama32_3b_layer"], rows_sample=1024, fused=fused)


@pytest.mark.parametrize("beta_path", [False, True])
def test_step_bf16_small(beta_path):
    """A bf16 step small enough to check every row: the one-call RoPE, split
    and plain VQ on the tensor cores, ragged tiles, the window rows."""
    w = synth.scaled(synth.WORKLOADS["llama32_3b_layer"], H=2, N=3001, K=300, W=200, M=512)
    _run(w, beta_path=beta_path)


def test_fused_and_separate_compositions_agree():
    """The fused composition (RoPE, split and plain VQ in one call, the
    retrieval rule after the split) and the separate one (RoPE and split on
    the second stream beside plain VQ) write the same step."""
    w = synth.scaled(synth.WORKLOADS["llama32_3b_layer"], H=4, N=8192, M=1024)
    k, c, Q = dev(synth.keys(w)), dev(synth.codebook(w)), dev(synth.queries(w))
    outs = []
    for fused in (True, False):
        step = A2ATSStep(w.B, w.H, w.N, w.d, w.K, torch.bfloat16, window=w.W,
                         fraction=w.fraction, rope_base=w.rope_base, M=w.M, fused=fused)
        step(k, c, queries=Q)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (step.k_tilde, step.count, step.perm, step.codes)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_step_is_deterministic():
    w = synth.scaled(synth.WORKLOADS["llama32_3b_layer"], N=8192, H=2, M=1024)
    k, c, Q = dev(synth.keys(w)), dev(synth.codebook(w)), dev(synth.queries(w))
    outs = []
    for _ in range(2):
        step = A2ATSStep(w.B, w.H, w.N, w.d, w.K, torch.bfloat16, window=w.W, fraction=w.fraction,
                         rope_base=w.rope_base, M=w.M)
        step(k, c, queries=Q)
        outs.append([t.clone() for t in (step.codes, step.perm, step.count, step.k_tilde,
                                         step.Hm, step.L)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_calibrated_steps_reuse_the_codebook_side():
    """calibrate() once, a first step that builds the codebook side, then
    steps that reuse it on new keys: the same codes, split and rotated keys as
    a step object that rebuilds everything for those keys."""
    w = synth.scaled(synth.WORKLOADS["llama32_3b_layer"], H=2, N=4096, K=256, W=128, M=1024)
    c, Q = dev(synth.codebook(w)), dev(synth.queries(w))
    mk = lambda: A2ATSStep(w.B, w.H, w.N, w.d, w.K, synth.DTYPES[w.dtype], window=w.W,
                           fraction=w.fraction, rope_base=w.rope_base, M=w.M, ridge=w.ridge)
    step = mk().calibrate(queries=Q)
    for i, seed in enumerate((0, 1, 2)):
        k = dev(synth.keys(w) if seed == 0 else synth.gaussian((w.B, w.H, w.N, w.d), seed=seed,
                                                                dtype=w.dtype))
        step(k, c, calibrated=True, reuse_codebook=i > 0)
        fresh = mk()
        fresh(k, c, queries=Q)
        torch.cuda.synchronize()
        assert torch.equal(step.L, fresh.L)
        assert torch.equal(step.count, fresh.count)
        assert torch.equal(step.perm, fresh.perm)
        assert torch.equal(step.k_tilde, fresh.k_tilde)
        assert torch.equal(step.codes, fresh.codes)
