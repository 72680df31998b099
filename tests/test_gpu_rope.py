"""GPU parity: windowed RoPE against the oracle (deploy-preview page,
paper-fidelity section, Eq. 11-12; v0.39.0 page, "How it works" step 4)."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_vq_gb300 as q
import synth
from _parity import assert_rows_close, assert_storage_close, dev, f64

pytestmark = pytest.mark.gpu
DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _oracle(k, lens, W, far, base, inter):
    B, H, N, d = k.shape
    x = f64(k)
    out = np.full((B, H, N, d), np.nan)
    for b in range(B):
        n = int(lens[b])
        pos = np.arange(n)
        for h in range(H):
            out[b, h, :n] = oracle.windowed_rope(x[b, h, :n], pos, n - 1, W, far, base, inter)
    return out


CASES = [
    # B, H, N, d, dtype, W, far, base, interleaved
    (2, 3, 300, 128, "bf16", 64, 0, 500000.0, False),
    (1, 2, 257, 128, "f32", 1000, 0, 10000.0, False),
    (2, 1, 130, 64, "f16", 16, 37, 10000.0, False),
    (1, 2, 100, 256, "bf16", 0, 0, 10000.0, False),
    (1, 1, 90, 32, "f32", 7, 5, 10000.0, True),
    (2, 2, 77, 24, "f32", 9, 0, 10000.0, False),
    (1, 1, 40, 8, "bf16", 3, 11, 100.0, True),
    # several 1024-row chunks per (b, h): chunks of far rows only beside the
    # chunk that holds the window, and far rows rotated by far_offset
    (2, 2, 2600, 128, "bf16", 100, 0, 500000.0, False),
    (2, 1, 2100, 64, "f16", 50, 7, 10000.0, False),
]


@pytest.mark.parametrize("case", CASES)
def test_rope_matches_oracle(case):
    B, H, N, d, dt, W, far, base, inter = case
    k = synth.gaussian((B, H, N, d), seed=N + d, dtype=dt, scale=3.0)
    lens = torch.tensor([N - 17 * b for b in range(B)], dtype=torch.int32)
    want = _oracle(k, lens.numpy(), W, far, base, inter)
    kd, ld = dev(k), dev(lens)
    # fp32 output: within 1e-3 of the row's max (contract), and far tighter in practice
    out = torch.full((B, H, N, d), 7.0, device="cuda")
    q.a2ats_windowed_rope(kd, window=W, far_offset=far, rope_base=base, interleaved=inter,
                          lengths=ld, out=out)
    got = f64(out)
    for b in range(B):
        n = int(lens[b])
        worst = assert_rows_close(got[b, :, :n].reshape(-1, d), want[b, :, :n].reshape(-1, d))
        assert worst < 2e-6
        assert (got[b, :, n:] == 7.0).all()  # rows past the length are untouched
    # half-precision storage output: at most one unit in the last place from
    # the oracle rounded to nearest even, plus the fp32 rotation's own error
    # (fp32 storage is the check above)
    if dt == "f32":
        return
    out2 = q.a2ats_windowed_rope(kd, window=W, far_offset=far, rope_base=base,
                                 interleaved=inter, lengths=ld)
    g2 = f64(out2)
    for b in range(B):
        n = int(lens[b])
        assert_storage_close(g2[b, :, :n], want[b, :, :n], DT[dt])


def test_far_rows_bit_equal_input_and_near_rows_rotated():
    k = synth.gaussian((1, 2, 500, 128), seed=3, dtype="bf16")
    out = q.a2ats_windowed_rope(dev(k), window=64, far_offset=0, rope_base=500000.0)
    o, x = out.cpu(), k
    assert torch.equal(o[:, :, :436], x[:, :, :436])
    assert not torch.equal(o[:, :, 436:], x[:, :, 436:])


def test_in_place_rotation():
    k = dev(synth.gaussian((1, 1, 200, 64), seed=4, dtype="f32"))
    ref = q.a2ats_windowed_rope(k, window=50, rope_base=10000.0)
    q.a2ats_windowed_rope(k, window=50, rope_base=10000.0, out=k)
    assert torch.equal(ref, k)


def test_empty_and_zero_length_sequences():
    k = dev(synth.gaussian((2, 1, 32, 16), seed=5, dtype="bf16"))
    out = torch.zeros_like(k)
    q.a2ats_windowed_rope(k, window=4, rope_base=10000.0, lengths=dev(torch.tensor([0, 32], dtype=torch.int32)), out=out)
    assert (out[0] == 0).all() and not (out[1] == 0).all()
    e = torch.empty((0, 8, 0, 128), dtype=torch.bfloat16, device="cuda")
    q.a2ats_windowed_rope(e, window=4, rope_base=10000.0)


@pytest.mark.parametrize("name", ["llama32_3b_layer"])
def test_rope_full_size_sampled(name):
    w = synth.WORKLOADS[name]
    k = synth.keys(w)
    out = q.a2ats_windowed_rope(dev(k), window=w.W, far_offset=w.far_offset,
                                rope_base=w.rope_base, out_dtype=torch.float32)
    rng = np.random.default_rng(0)
    N = w.N
    for b in range(w.B):
        for h in range(w.H):
            rows = np.unique(np.concatenate([rng.choice(N, 256, replace=False),
                                             np.arange(N - w.W - 2, N)]))
            want = oracle.windowed_rope(k[b, h, rows], rows, N - 1, w.W, w.far_offset, w.rope_base)
            worst = assert_rows_close(f64(out[b, h, rows]), want)
            assert worst < 2e-6
