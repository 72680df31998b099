"""The allocation-free retrieval split gives the same result as the workspace
version.

a2ats_select_retrieval_set_static serves callers that cannot allocate device
memory (their pool belongs to another allocator, or their path must never risk
an allocation): its scratch is a fixed array inside the library.  This test
calls it through the C ABI twice in a row -- the second call runs on scratch
the first one left behind -- and checks each result against
a2ats_select_retrieval_set with a caller workspace.  It also checks that a
shape beyond the fixed array is refused before anything runs.  The file name
sorts last so a stop-at-first-failure run has run every other test first.
"""
import ctypes

import pytest
import torch

import query_aware_vq_gb300 as q
import synth

pytestmark = pytest.mark.gpu

_P = ctypes.c_void_p
_I32, _I64, _D = ctypes.c_int32, ctypes.c_int64, ctypes.c_double


def _static_fn():
    fn = q.library().a2ats_select_retrieval_set_static
    fn.argtypes = [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _D, _P, _P, _P, _P]
    fn.restype = ctypes.c_int
    return fn


_DT = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}


def _call_static(keys, lengths, fraction, rope):
    B, H, N, d = keys.shape
    perm = torch.full((B, H, N), -1, dtype=torch.int32, device="cuda")
    count = torch.full((B, H), -1, dtype=torch.int32, device="cuda")
    status = _static_fn()(keys.data_ptr(), _DT[keys.dtype], B, H, N, d,
                          lengths.data_ptr() if lengths is not None else None, None, fraction,
                          ctypes.byref(rope) if rope is not None else None, perm.data_ptr(),
                          count.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert status == 0, q.library().a2ats_status_string(status)
    return perm, count


def test_static_split_matches_workspace_split_twice():
    w = synth.scaled(synth.WORKLOADS["llama32_3b_layer"], B=2, H=4, N=20000)
    keys = synth.keys(w).cuda()
    lengths = torch.tensor([20000, 17321], dtype=torch.int32, device="cuda")
    rope = q.RopeParams(w.W, 0, w.rope_base, 0)
    want_perm, want_count = q.a2ats_select_retrieval_set(keys, None, w.fraction, lengths=lengths,
                                                         rope=rope)
    for _ in range(2):
        perm, count = _call_static(keys, lengths, w.fraction, rope)
        torch.cuda.synchronize()
        assert torch.equal(count, want_count)
        for b in range(w.B):
            n = int(lengths[b])
            assert torch.equal(perm[b, :, :n], want_perm[b, :, :n])


@pytest.mark.parametrize("B,H,N,d,dt,with_rope", [
    # exactly at the key limit (the last slot of the score region), widest rows
    (1, 8, 131072, 256, "f16", True),
    # no fused rotation, fp32 keys, ragged lengths
    (3, 5, 5000, 64, "f32", False),
])
def test_static_split_at_the_limits_matches_workspace_split(B, H, N, d, dt, with_rope):
    keys = synth.gaussian((B, H, N, d), seed=N + d, dtype=dt).cuda()
    lengths = torch.tensor([N - 999 * b for b in range(B)], dtype=torch.int32, device="cuda")
    rope = q.RopeParams(300, 0, 10000.0, 0) if with_rope else None
    want_perm, want_count = q.a2ats_select_retrieval_set(keys, None, 0.1, lengths=lengths,
                                                         rope=rope)
    for _ in range(2):
        perm, count = _call_static(keys, lengths, 0.1, rope)
        torch.cuda.synchronize()
        assert torch.equal(count, want_count)
        for b in range(B):
            n = int(lengths[b])
            assert torch.equal(perm[b, :, :n], want_perm[b, :, :n])


def test_static_split_refuses_too_many_heads():
    B, H, N, d = 1, 1025, 4, 64
    keys = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    perm = torch.empty((B, H, N), dtype=torch.int32, device="cuda")
    count = torch.empty((B, H), dtype=torch.int32, device="cuda")
    status = _static_fn()(keys.data_ptr(), 1, B, H, N, d, None, None, 0.1, None,
                          perm.data_ptr(), count.data_ptr(), None)
    assert status == -7


def test_static_split_refuses_shapes_beyond_its_array():
    keys = torch.zeros((1, 8, 200000, 128), dtype=torch.bfloat16, device="cuda")
    perm = torch.empty((1, 8, 200000), dtype=torch.int32, device="cuda")
    count = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    status = _static_fn()(keys.data_ptr(), 1, 1, 8, 200000, 128, None, None, 0.1, None,
                          perm.data_ptr(), count.data_ptr(), None)
    assert status == -7
