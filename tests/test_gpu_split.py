"""GPU parity: retrieval split against the oracle (API page,
a2ats_select_retrieval_set): exact size ceil(fraction * n), disjoint and
covering halves in ascending order, membership equal to the oracle's except
for rows within 1e-5 of the threshold score."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import check_split, dev, f64

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, N, d, dtype, fraction, query mode, rope
    (2, 3, 1000, 128, "bf16", 0.1, "proxy", dict(window=64, rope_base=500000.0)),
    (1, 2, 5000, 128, "f32", 0.05, "given", None),
    (2, 1, 777, 64, "f16", 0.2, "proxy", dict(window=16, far_offset=5, rope_base=10000.0)),
    (1, 1, 3000, 256, "bf16", 1.0, "given", None),
    (1, 2, 300, 24, "f32", 0.3, "proxy", dict(window=8, rope_base=10000.0)),
    (1, 1, 10, 16, "bf16", 0.0, "proxy", None),
    (1, 1, 1, 16, "bf16", 0.5, "proxy", None),
    (1, 1, 70000, 128, "bf16", 0.02, "proxy", dict(window=100, rope_base=500000.0)),
    # segments too long for the select kernel's shared-memory cache
    (1, 1, 140000, 16, "bf16", 0.03, "proxy", None),
    # many (b, h): the select's smaller CTAs
    (16, 8, 300, 64, "bf16", 0.1, "proxy", dict(window=32, rope_base=500000.0)),
]


@pytest.mark.parametrize("case", CASES)
def test_split_matches_oracle(case):
    B, H, N, d, dt, f, qmode, rope = case
    k = synth.gaussian((B, H, N, d), seed=N, dtype=dt)
    lens = torch.tensor([max(N - 13 * b, 0) for b in range(B)], dtype=torch.int32)
    query = synth.gaussian((B, H, d), seed=N + 1, dtype=dt) if qmode == "given" else None
    perm, count = q.a2ats_select_retrieval_set(dev(k), dev(query) if query is not None else None,
                                               f, lengths=dev(lens), rope=rope)
    perm, count = perm.cpu().numpy(), count.cpu().numpy()
    for b in range(B):
        n = int(lens[b])
        for h in range(H):
            v = f64(k[b, h, :n])
            if rope is not None:
                v = oracle.windowed_rope(v, np.arange(n), n - 1, rope["window"],
                                         rope.get("far_offset", 0), rope["rope_base"])
            qv = f64(query[b, h]) if query is not None else v[n - 1]
            _, cnt, scores, kth = oracle.select_retrieval_set(v, qv, f)
            check_split(perm[b, h], int(count[b, h]), n, cnt, scores, kth)


def test_equal_scores_keep_lowest_indices():
    k = torch.ones((1, 1, 4096, 16), dtype=torch.bfloat16)
    perm, count = q.a2ats_select_retrieval_set(dev(k), None, 0.25)
    c = int(count[0, 0])
    assert c == 1024
    assert perm[0, 0, :c].cpu().tolist() == list(range(1024))


def test_proxy_row_always_retrieved():
    k = synth.gaussian((1, 4, 2000, 128), seed=5, dtype="bf16")
    perm, count = q.a2ats_select_retrieval_set(dev(k), None, 0.01,
                                               rope=dict(window=64, rope_base=500000.0))
    for h in range(4):
        assert 1999 in perm[0, h, :int(count[0, h])].cpu().tolist()


@pytest.mark.parametrize("name", ["llama32_3b_layer"])
def test_split_full_size(name):
    w = synth.WORKLOADS[name]
    k = synth.keys(w)
    rope = dict(window=w.W, far_offset=w.far_offset, rope_base=w.rope_base)
    perm, count = q.a2ats_select_retrieval_set(dev(k), None, w.fraction, rope=rope)
    perm, count = perm.cpu().numpy(), count.cpu().numpy()
    for b in range(w.B):
        for h in range(w.H):
            v = oracle.windowed_rope(k[b, h], np.arange(w.N), w.N - 1, w.W, 0, w.rope_base)
            _, cnt, scores, kth = oracle.select_retrieval_set(v, v[-1], w.fraction)
            check_split(perm[b, h], int(count[b, h]), w.N, cnt, scores, kth)


@pytest.mark.parametrize("case", [
    # B, H, N, d, dtype, out dtype, fraction, rope
    (2, 3, 1000, 128, "bf16", "bf16", 0.1, dict(window=64, rope_base=500000.0)),
    (1, 2, 777, 64, "f16", "f32", 0.2, dict(window=16, far_offset=5, rope_base=10000.0)),
    (2, 1, 300, 128, "bf16", "bf16", 0.3, dict(window=40, rope_base=10000.0, interleaved=1)),
    (1, 2, 300, 24, "f32", "f32", 0.3, dict(window=8, rope_base=10000.0)),   # no fused form
    (1, 1, 5, 16, "bf16", "bf16", 0.5, dict(window=2, rope_base=10000.0)),
    # several 1024-row chunks per (b, h): chunks of far rows only (copied
    # as loaded, or converted) beside the chunk that holds the window
    (2, 2, 2600, 128, "bf16", "bf16", 0.1, dict(window=64, rope_base=500000.0)),
    (1, 1, 2600, 128, "bf16", "f32", 0.1, dict(window=64, rope_base=500000.0)),
    (1, 1, 2100, 64, "f16", "f16", 0.2, dict(window=16, far_offset=5, rope_base=10000.0)),
])
def test_rotated_split_equals_the_two_calls(case):
    """The one-pass call writes exactly what a2ats_windowed_rope and
    a2ats_select_retrieval_set(rope=...) write, ragged lengths included."""
    B, H, N, d, dt, odt, f, rope = case
    k = dev(synth.gaussian((B, H, N, d), seed=N + 7, dtype=dt))
    lens = dev(torch.tensor([max(N - 17 * b, 1) for b in range(B)], dtype=torch.int32))
    want_out = torch.zeros((B, H, N, d), dtype=synth.DTYPES[odt], device="cuda")
    q.a2ats_windowed_rope(k, lengths=lens, out=want_out, **rope)
    want_perm, want_count = q.a2ats_select_retrieval_set(k, None, f, lengths=lens, rope=rope)
    out = torch.zeros_like(want_out)
    out, perm, count = q.a2ats_select_retrieval_set_rotated(k, None, f, rope=rope, lengths=lens,
                                                            out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, want_out)
    assert torch.equal(count, want_count)
    for b in range(B):
        n = int(lens[b])
        assert torch.equal(perm[b, :, :n], want_perm[b, :, :n])


def test_copy_retrieval_rows_touches_only_the_retrieval_rows():
    B, H, N = 2, 3, 500
    k = dev(synth.gaussian((B, H, N, 64), seed=3, dtype="bf16"))
    lens = dev(torch.tensor([N, 321], dtype=torch.int32))
    perm, count = q.a2ats_select_retrieval_set(k, None, 0.1, lengths=lens)
    src = torch.arange(B * H * N, dtype=torch.int32, device="cuda").reshape(B, H, N)
    dst = torch.full((B, H, N), -1, dtype=torch.int32, device="cuda")
    q.a2ats_copy_retrieval_rows(src, dst, perm, count, lengths=lens)
    want = torch.full_like(dst, -1)
    for b in range(B):
        for h in range(H):
            sel = perm[b, h, :int(count[b, h])].long()
            want[b, h, sel] = src[b, h, sel]
    assert torch.equal(dst, want)
