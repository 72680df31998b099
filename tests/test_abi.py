"""The C-ABI library builds for sm_103a, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch
(CPU only: nothing here reaches a kernel)."""
import ctypes

import pytest

import query_aware_vq_gb300 as q
from query_aware_vq_gb300 import build as qbuild


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return q.library()


def test_every_declared_symbol_is_exported(lib):
    names = q.declared_symbols()
    assert len(names) >= 12
    for n in ("a2ats_query_second_moment", "a2ats_cholesky_factor", "a2ats_windowed_rope",
              "a2ats_h_weighted_assign", "a2ats_query_aware_assign",
              "a2ats_select_retrieval_set"):
        assert n in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert lib.a2ats_status_string(0) == b"A2ATS_OK"
    assert lib.a2ats_status_string(-2) == b"A2ATS_ERR_SHAPE"
    assert lib.a2ats_status_string(-6) == b"A2ATS_ERR_WORKSPACE"
    assert lib.a2ats_status_string(12345) == b"A2ATS_ERR_UNKNOWN"


def test_workspace_sizes_grow_with_shape(lib):
    a = lib.a2ats_h_weighted_assign_workspace_size(1, 8, 32768, 128, 1024)
    b = lib.a2ats_h_weighted_assign_workspace_size(1, 8, 32768, 128, 4096)
    assert 0 < a < b
    assert lib.a2ats_select_retrieval_set_workspace_size(1, 8, 32768, 128) >= 8 * 32768 * 4
    assert lib.a2ats_query_second_moment_workspace_size(8, 8192, 128) >= 8 * 128 * 128 * 4


FAKE = 0x1000  # a 16-byte aligned address that is never dereferenced


def _rope(window=64, far=0, base=10000.0, inter=0):
    return ctypes.byref(q.RopeParams(window, far, base, inter))


def test_rope_validation(lib):
    f = lib.a2ats_windowed_rope
    assert f(FAKE, 7, FAKE, 0, 1, 1, 16, 128, None, _rope(), None) == -3      # dtype
    assert f(FAKE, 1, FAKE, 1, 1, 1, 16, 130, None, _rope(), None) == -2      # d % 8
    assert f(FAKE, 1, FAKE, 1, 1, 1, 16, 264, None, _rope(), None) == -2      # d > 256
    assert f(FAKE, 1, FAKE, 1, 1, 1, 1 << 24, 128, None, _rope(), None) == -2  # positions
    assert f(FAKE, 1, FAKE, 1, 1, 1, 16, 128, None, None, None) == -1          # no params
    assert f(FAKE, 1, FAKE, 1, 1, 1, 16, 128, None, _rope(base=-1.0), None) == -1
    assert f(FAKE + 8, 1, FAKE, 1, 1, 1, 16, 128, None, _rope(), None) == -4   # alignment
    assert f(None, 1, FAKE, 1, 1, 1, 16, 128, None, _rope(), None) == -1
    assert f(FAKE, 1, FAKE, 0, 1, 1, 16, 128, None, _rope(), None) == -1      # alias, dtypes differ
    assert f(None, 1, None, 1, 0, 1, 16, 128, None, _rope(), None) == 0       # empty: no-op


def test_assign_validation(lib):
    f = lib.a2ats_h_weighted_assign
    args = lambda **kw: [kw.get("x", FAKE), kw.get("dt", 1), 1, 2, 64, kw.get("d", 128), None,
                         FAKE, kw.get("K", 16), None, None, kw.get("rows", 0), kw.get("perm"),
                         kw.get("count"), FAKE, kw.get("ws", FAKE), kw.get("wsb", 1 << 30), None]
    assert f(*args(dt=9)) == -3
    assert f(*args(K=0)) == -2
    assert f(*args(d=12)) == -2
    assert f(*args(rows=5)) == -1
    assert f(*args(rows=1)) == -1                  # retrieval rows need perm and count
    assert f(*args(x=FAKE + 4)) == -4
    assert f(*args(ws=None)) == -6
    assert f(*args(wsb=16)) == -6
    for g in (lib.a2ats_query_aware_assign, lib.a2ats_query_aware_assign_reuse):
        base = [FAKE, 1, 1, 2, 64, 128, None, FAKE, 16, None]
        tail = [None, 0, None, None, FAKE, FAKE, 1 << 30, None]
        for beta in (-0.1, 1.5, float("nan")):
            assert g(*base, beta, *tail) == -1
        assert g(*base, 0.5, None, 0, None, None, FAKE, None, 0, None) == -6  # no workspace


def test_split_and_calibration_validation(lib):
    s = lib.a2ats_select_retrieval_set
    for frac in (-0.01, 1.01, float("nan")):
        assert s(FAKE, 1, 1, 2, 64, 128, None, None, frac, None, FAKE, FAKE, FAKE, 1 << 30,
                 None) == -1
    assert s(FAKE, 1, 1, 2, 64, 128, None, None, 0.2, None, FAKE, FAKE, None, 0, None) == -6
    m = lib.a2ats_query_second_moment
    assert m(FAKE, 1, 2, 0, 128, 1e-4, FAKE, FAKE, 1 << 30, None) == -2       # M = 0
    assert m(FAKE, 1, 2, 10, 128, -1.0, FAKE, FAKE, 1 << 30, None) == -1      # ridge < 0
    assert m(FAKE, 1, 2, 10, 128, 1e-4, FAKE, None, 0, None) == -6
    c = lib.a2ats_cholesky_factor
    assert c(FAKE, 2, 100, FAKE, FAKE, None) == -2
    assert c(FAKE, 2, 128, FAKE, None, None) == -1


def test_rotated_split_validation(lib):
    r = lib.a2ats_select_retrieval_set_rotated
    rope = q.RopeParams(64, 0, 500000.0, 0)
    ws = 1 << 30
    # rope is required, k_out may not alias keys, the out dtype is checked
    assert r(FAKE, 1, 1, 2, 64, 128, None, None, 0.2, None, FAKE + 4096, 1, FAKE, FAKE, FAKE,
             ws, None) == -1
    assert r(FAKE, 1, 1, 2, 64, 128, None, None, 0.2, ctypes.byref(rope), FAKE, 1, FAKE, FAKE,
             FAKE, ws, None) == -1
    assert r(FAKE, 1, 1, 2, 64, 128, None, None, 0.2, ctypes.byref(rope), FAKE + 4096, 7, FAKE,
             FAKE, FAKE, ws, None) == -3
    assert r(FAKE, 1, 1, 2, 64, 128, None, None, 1.5, ctypes.byref(rope), FAKE + 4096, 1, FAKE,
             FAKE, FAKE, ws, None) == -1
    assert r(FAKE, 1, 1, 2, 64, 128, None, None, 0.2, ctypes.byref(rope), FAKE + 4100, 1, FAKE,
             FAKE, FAKE, ws, None) == -4
    assert r(FAKE, 1, 1, 2, 64, 128, None, None, 0.2, ctypes.byref(rope), FAKE + 4096, 1, FAKE,
             FAKE, None, 0, None) == -6


def test_rope_split_plain_assign_validation(lib):
    f = lib.a2ats_rope_split_plain_assign
    rope = q.RopeParams(64, 0, 500000.0, 0)
    ws = 1 << 30

    def call(keys=FAKE, dt=1, K=256, k_out=FAKE + 4096, codes=FAKE + 8192, rp=rope, frac=0.2,
             ws_ptr=FAKE, nb=ws, codebook=FAKE + 12288, split_stream=None):
        return f(keys, dt, 1, 2, 64, 128, None, None, frac,
                 ctypes.byref(rp) if rp is not None else None, codebook, K, k_out, FAKE, FAKE,
                 codes, 0, None, split_stream, ws_ptr, nb, None)

    assert call(rp=None) == -1                 # rope is required
    assert call(k_out=FAKE) == -1              # k_out may not alias keys
    assert call(dt=7) == -3
    assert call(K=0) == -2
    assert call(frac=-0.1) == -1
    assert call(codes=None) == -1
    assert call(codebook=FAKE + 12290) == -4   # misaligned codebook
    assert call(split_stream=FAKE) == -1       # a split stream needs split_done
    assert call(ws_ptr=None, nb=0) == -6
    # the workspace holds both the assignment's and the split's
    need = lib.a2ats_rope_split_plain_assign_workspace_size(1, 2, 64, 128, 256)
    assert need > lib.a2ats_h_weighted_assign_workspace_size(1, 2, 64, 128, 256)
    assert need > lib.a2ats_select_retrieval_set_workspace_size(1, 2, 64, 128)
    assert call(nb=need - 1) == -6


def test_code_attention_topk_validation(lib):
    f = lib.a2ats_code_attention_topk
    rope = q.RopeParams(64, 0, 500000.0, 0)
    ws = 1 << 30

    def call(dt=1, K=256, rp=rope, far_b=2048, frac=0.1, codes=FAKE + 4096, query=FAKE + 8192,
             ws_ptr=FAKE, nb=ws):
        return f(FAKE, dt, 1, 2, 64, 128, None, codes, FAKE + 12288, K, query,
                 ctypes.byref(rp) if rp is not None else None, far_b, frac, FAKE + 16384,
                 FAKE + 20480, FAKE, ws_ptr, nb, None)

    assert call(rp=None) == -1
    assert call(dt=5) == -3
    assert call(K=0) == -2
    assert call(frac=1.5) == -1
    assert call(far_b=1 << 24) == -1
    assert call(codes=None) == -1
    assert call(query=FAKE + 8196) == -4
    assert call(ws_ptr=None, nb=0) == -6
    need = lib.a2ats_code_attention_topk_workspace_size(1, 2, 64, 128, 256)
    assert need >= 4 * (2 * 128 + 2 * 256)
    assert call(nb=need - 1) == -6


def test_dequantize_validation(lib):
    f = lib.a2ats_dequantize
    assert f(FAKE, FAKE + 4096, 9, 1, 2, 64, 128, 256, None, FAKE + 8192, None) == -3
    assert f(FAKE, FAKE + 4096, 1, 1, 2, 64, 12, 256, None, FAKE + 8192, None) == -2
    assert f(FAKE, FAKE + 4096, 1, 1, 2, 64, 128, 0, None, FAKE + 8192, None) == -2
    assert f(None, FAKE + 4096, 1, 1, 2, 64, 128, 256, None, FAKE + 8192, None) == -1
    assert f(FAKE, FAKE + 4096, 1, 1, 2, 64, 128, 256, None, FAKE + 4096, None) == -1
    assert f(FAKE, FAKE + 4100, 1, 1, 2, 64, 128, 256, None, FAKE + 8192, None) == -4
    assert f(None, None, 1, 0, 2, 64, 128, 256, None, None, None) == 0


def test_byte_accounting_matches_the_page_table():
    """v0.39.0 page, "What you get with the defaults", through the C ABI, and
    the same figures as the oracle's accounting."""
    import oracle
    from _golden import lines
    for row in lines("compression_defaults.txt"):
        acc = q.a2ats_byte_accounting(1000, 128, int(row[0]), int(row[1]))
        assert acc["assigned_avg_bits"] == float(row[2])
        assert acc["compression_ratio"] == float(row[3])
        assert acc["codebook_bytes"] / 1024 == float(row[4])
        assert acc == oracle.byte_accounting(1000, 128, int(row[0]), int(row[1]))
    # the full-width codes of the Llama-3.2-3B layer: 10 bits per 128-number key
    acc = q.a2ats_byte_accounting(32768, 128, 128, 10)
    assert acc["compressed_key_bytes"] == acc["compressed_value_bytes"] == 32768 * 10 / 8
    assert acc["compression_ratio"] == 16 * 128 / 10
    assert q.a2ats_byte_accounting(0, 128, 8, 8)["compression_ratio"] == 16.0
    with pytest.raises(q.A2ATSError):
        q.a2ats_byte_accounting(10, 128, 5, 8)


def test_copy_retrieval_rows_validation(lib):
    f = lib.a2ats_copy_retrieval_rows
    assert f(FAKE, FAKE, -1, 2, 10, None, FAKE, FAKE, None) == -2
    assert f(FAKE, FAKE, 1, 70000, 10, None, FAKE, FAKE, None) == -2
    assert f(None, FAKE, 1, 2, 10, None, FAKE, FAKE, None) == -1
    assert f(FAKE, FAKE, 1, 2, 10, None, None, FAKE, None) == -1
    assert f(None, None, 0, 2, 10, None, None, None, None) == 0


def test_cholesky_rows_validation(lib):
    f = lib.a2ats_cholesky_rows
    ws = lib.a2ats_cholesky_rows_workspace_size(2, 100, 64)
    assert ws >= 2 * (2 * 64 * 64 + 100) * 4
    W = FAKE + (1 << 24)
    assert f(FAKE, 9, 2, 100, 64, FAKE + 65536, FAKE + 131072, W, ws, None) == -3
    assert f(FAKE, 1, 2, 100, 12, FAKE + 65536, FAKE + 131072, W, ws, None) == -2
    assert f(FAKE, 1, 2, 1 << 24, 64, FAKE + 65536, FAKE + 131072, W, ws, None) == -2
    assert f(None, 1, 2, 100, 64, FAKE + 65536, FAKE + 131072, W, ws, None) == -1
    assert f(FAKE, 0, 2, 100, 64, FAKE + 65536, FAKE, W, ws, None) == -1
    assert f(FAKE + 8, 1, 2, 100, 64, FAKE + 65536, FAKE + 131072, W, ws, None) == -4
    assert f(FAKE, 1, 2, 100, 64, FAKE + 65536, FAKE + 131072, W, ws - 1, None) == -6
    assert f(FAKE, 1, 2, 100, 64, FAKE + 65536, FAKE + 131072, None, ws, None) == -6
    assert f(None, 1, 0, 100, 64, None, None, None, 0, None) == 0


def test_cholesky_solve_rows_validation(lib):
    f = lib.a2ats_cholesky_solve_rows
    assert f(FAKE, 2, 100, 12, FAKE + 65536, FAKE, None) == -2
    assert f(FAKE, 4096, 1 << 24, 64, FAKE + 65536, FAKE, None) == -2
    assert f(None, 2, 100, 64, FAKE + 65536, FAKE, None) == -1
    assert f(FAKE, 2, 100, 64, None, FAKE, None) == -1
    assert f(FAKE, 2, 100, 64, FAKE + 65540, FAKE, None) == -4
    assert f(None, 2, 0, 64, None, None, None) == 0


def test_kmeanspp_validation(lib):
    f = lib.a2ats_kmeanspp
    H, n, d, K = 2, 100, 8, 4
    ws = lib.a2ats_kmeanspp_workspace_size(H, n, d, K)
    assert ws >= (H * n + H * K) * 8 + lib.a2ats_h_weighted_assign_workspace_size(1, H, n, d, K)
    z, u, c, k, o, W = (FAKE, FAKE + 65536, FAKE + 131072, FAKE + 196608, FAKE + 262144,
                        FAKE + (1 << 24))
    assert f(z, H, n, 12, K, u, 3, c, k, o, W, ws, None) == -2
    assert f(z, H, n, d, 0, u, 3, c, k, o, W, ws, None) == -2
    assert f(z, H, 0, d, K, u, 3, c, k, o, W, ws, None) == -2
    assert f(z, H, n, d, K, u, -1, c, k, o, W, ws, None) == -1
    assert f(z, H, n, d, K, None, 3, c, k, o, W, ws, None) == -1
    assert f(z, H, n, d, K, u + 4, 3, c, k, o, W, ws, None) == -4
    assert f(z, H, n, d, K, u, 3, c + 8, k, o, W, ws, None) == -4
    # z [H, n, d] fp32 spans 6400 bytes: centroids 1 KB in overlap it
    assert f(z, H, n, d, K, u, 3, z + 1024, k, o, W, ws, None) == -1
    assert f(z, H, n, d, K, u, 3, c, c + 128, o, W, ws, None) == -1
    assert f(z, H, n, d, K, u, 3, c, k, o, W, ws - 1, None) == -6
    assert f(None, 0, n, d, K, None, 3, None, None, None, None, 0, None) == 0


def test_subvector_assign_validation(lib):
    f = lib.a2ats_subvector_assign
    B, H, N, d, s, K = 1, 2, 64, 128, 8, 256
    ws = lib.a2ats_subvector_assign_workspace_size(B, H, N, d, s, K)
    assert ws >= (2 * H * K * s + H * K) * 4 + B * H * N
    x, c, L, p, n, k, W = (FAKE, FAKE + 65536, FAKE + 131072, FAKE + 196608, FAKE + 262144,
                           FAKE + 327680, FAKE + (1 << 24))
    assert f(x, 9, B, H, N, d, None, s, c, K, L, p, n, k, W, ws, None) == -3
    assert f(x, 1, B, H, N, d, None, 12, c, K, L, p, n, k, W, ws, None) == -2
    assert f(x, 1, B, H, N, 24, None, 16, c, K, L, p, n, k, W, ws, None) == -2
    assert f(x, 1, B, H, N, d, None, s, c, 1025, L, p, n, k, W, ws, None) == -2
    assert f(x, 1, B, H, N, d, None, s, c, K, L, p, None, k, W, ws, None) == -1
    assert f(x, 1, B, H, N, d, None, s, None, K, L, p, n, k, W, ws, None) == -1
    assert f(x, 1, B, H, N, d, None, s, c + 4, K, L, p, n, k, W, ws, None) == -4
    assert f(x, 1, B, H, N, d, None, s, c, K, L + 8, p, n, k, W, ws, None) == -4
    assert f(x, 1, B, H, N, d, None, s, c, K, L, p, n, k, W, ws - 1, None) == -6
    assert f(None, 1, 0, H, N, d, None, s, None, K, None, None, None, None, None, 0, None) == 0


def test_subvector_query_aware_assign_validation(lib):
    f = lib.a2ats_subvector_query_aware_assign
    B, H, N, d, s, K = 1, 2, 64, 128, 8, 256
    ws = lib.a2ats_subvector_query_aware_assign_workspace_size(B, H, N, d, s, K)
    assert ws >= (H * K * s + 2 * H * K) * 4 + B * H * N
    x, c, q_, p, n, k, W = (FAKE, FAKE + 65536, FAKE + 131072, FAKE + 196608, FAKE + 262144,
                            FAKE + 327680, FAKE + (1 << 24))
    assert f(x, 9, B, H, N, d, None, s, c, K, q_, 0.5, p, n, k, W, ws, None) == -3
    assert f(x, 1, B, H, N, d, None, 12, c, K, q_, 0.5, p, n, k, W, ws, None) == -2
    assert f(x, 1, B, H, N, d, None, s, c, 2048, q_, 0.5, p, n, k, W, ws, None) == -2
    assert f(x, 1, B, H, N, d, None, s, c, K, q_, 1.5, p, n, k, W, ws, None) == -1
    assert f(x, 1, B, H, N, d, None, s, c, K, q_, float("nan"), p, n, k, W, ws, None) == -1
    assert f(x, 1, B, H, N, d, None, s, c, K, q_, 0.5, None, n, k, W, ws, None) == -1
    assert f(x, 1, B, H, N, d, None, s, c, K, q_ + 4, 0.5, p, n, k, W, ws, None) == -4
    assert f(x, 1, B, H, N, d, None, s, c, K, q_, 0.5, p, n, k, W, ws - 1, None) == -6
    assert f(None, 1, B, 0, N, d, None, s, None, K, None, 0.5, None, None, None, None, 0,
             None) == 0


def test_binding_signatures_match_the_header():
    """Every call the binding declares has as many arguments as its
    prototype in include/a2ats.h (the binding passes plain ctypes values, so
    a drift would go unnoticed until a call misbehaves)."""
    import re
    with open(q.HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(?:int|size_t|uint64_t|double|const char\*)\s+(a2ats_\w+)\s*"
                         r"\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        protos[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    assert set(protos) == set(q.declared_symbols())
    for name, args in q._SIGS.items():
        assert protos[name] == len(args), name


def test_binding_refuses_strided_and_host_tensors():
    """The binding hands data pointers to the library: a tensor that is not
    row-major contiguous, or not on a CUDA device, is refused before any
    call."""
    import torch
    codes = torch.zeros((1, 2, 8), dtype=torch.int32)
    cb = torch.zeros((2, 4, 16), dtype=torch.float32)
    with pytest.raises(ValueError, match="contiguous"):
        q.a2ats_dequantize(codes.transpose(1, 2), cb)
    with pytest.raises(ValueError, match="CUDA"):
        q.a2ats_dequantize(codes, cb)
