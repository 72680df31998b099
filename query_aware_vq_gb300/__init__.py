"""Python binding of liba2ats.so -- the GB300 (sm_103a) library for the hot
path of A2ATS-style retrieval-based KV-cache compression.

Every function here has the name of the C entry point it wraps (see
include/a2ats.h) and only marshals arguments: tensor pointers, sizes, the
current CUDA stream, and a scratch workspace tensor when the caller gives none.
All arithmetic runs in the library's CUDA kernels.  There is no CPU path: the
functions raise when the library is missing or a tensor is not a contiguous
tensor on a CUDA device.

Layouts: keys [B, H, N, d] (a 2-D [N, d] array is taken as B = H = 1),
codebooks [H, K, d], H / L matrices [H, d, d] fp32, per-(b, h) queries
[B, H, d]; dtypes fp32, bf16 or fp16.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liba2ats.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "a2ats.h")

A2ATS_ROWS = {"all": 0, "retrieval": 1, "bulk": 2, "last": 3}
_DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}


class A2ATSError(RuntimeError):
    """A non-zero status from the library."""

    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        name = _load().a2ats_status_string(status).decode()
        super().__init__(f"{fn}: {name} ({status}){': ' + detail if detail else ''}")


class RopeParams(ctypes.Structure):
    """a2ats_rope_params: windowed RoPE (window, far_offset, base, pairing)."""

    _fields_ = [("window", ctypes.c_int32), ("far_offset", ctypes.c_int32),
                ("rope_base", ctypes.c_double), ("interleaved", ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I32, _I64, _D, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_size_t
_SIGS = {
    "a2ats_windowed_rope": [_P, _I32, _P, _I32, _I64, _I64, _I64, _I64, _P, _P, _P],
    "a2ats_append_rows": [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _P],
    "a2ats_query_second_moment_workspace_size": [_I64, _I64, _I64],
    "a2ats_query_second_moment": [_P, _I32, _I64, _I64, _I64, _D, _P, _P, _SZ, _P],
    "a2ats_cholesky_factor": [_P, _I64, _I64, _P, _P, _P],
    "a2ats_h_weighted_assign_workspace_size": [_I64, _I64, _I64, _I64, _I64],
    "a2ats_h_weighted_assign": [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _I64, _P, _P, _I32, _P,
                                _P, _P, _P, _SZ, _P],
    "a2ats_h_weighted_assign_reuse": [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _I64, _P, _P,
                                      _I32, _P, _P, _P, _P, _SZ, _P],
    "a2ats_query_aware_assign_workspace_size": [_I64, _I64, _I64, _I64, _I64],
    "a2ats_query_aware_assign": [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _I64, _P, _D, _P,
                                 _I32, _P, _P, _P, _P, _SZ, _P],
    "a2ats_query_aware_assign_reuse": [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _I64, _P, _D,
                                       _P, _I32, _P, _P, _P, _P, _SZ, _P],
    "a2ats_select_retrieval_set_workspace_size": [_I64, _I64, _I64, _I64],
    "a2ats_select_retrieval_set": [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _D, _P, _P, _P, _P,
                                   _SZ, _P],
    "a2ats_select_retrieval_set_rotated": [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _D, _P, _P,
                                           _I32, _P, _P, _P, _SZ, _P],
    "a2ats_copy_retrieval_rows": [_P, _P, _I64, _I64, _I64, _P, _P, _P, _P],
    "a2ats_rope_split_plain_assign_workspace_size": [_I64, _I64, _I64, _I64, _I64],
    "a2ats_code_attention_topk_workspace_size": [_I64, _I64, _I64, _I64, _I64],
    "a2ats_dequantize": [_P, _P, _I32, _I64, _I64, _I64, _I64, _I64, _P, _P, _P],
    "a2ats_byte_accounting": [_I64, _I64, _I64, _I32, _P],
    "a2ats_code_attention_topk": [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _P,
                                  _I32, _D, _P, _P, _P, _P, _SZ, _P],
    "a2ats_rope_split_plain_assign": [_P, _I32, _I64, _I64, _I64, _I64, _P, _P, _D, _P, _P,
                                      _I64, _P, _P, _P, _P, _I32, _P, _P, _P, _SZ, _P],
    "a2ats_cholesky_rows_workspace_size": [_I64, _I64, _I64],
    "a2ats_cholesky_rows": [_P, _I32, _I64, _I64, _I64, _P, _P, _P, _SZ, _P],
    "a2ats_cholesky_solve_rows": [_P, _I64, _I64, _I64, _P, _P, _P],
    "a2ats_kmeanspp_workspace_size": [_I64, _I64, _I64, _I64],
    "a2ats_kmeanspp": [_P, _I64, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P, _SZ, _P],
    "a2ats_subvector_assign_workspace_size": [_I64, _I64, _I64, _I64, _I64, _I64],
    "a2ats_subvector_assign": [_P, _I32, _I64, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _P,
                               _P, _P, _P, _SZ, _P],
    "a2ats_subvector_query_aware_assign_workspace_size": [_I64, _I64, _I64, _I64, _I64, _I64],
    "a2ats_subvector_query_aware_assign": [_P, _I32, _I64, _I64, _I64, _I64, _P, _I64, _P, _I64,
                                           _P, _D, _P, _P, _P, _P, _SZ, _P],
    "a2ats_status_string": [_I32],
    "a2ats_last_error": [],
    "a2ats_kernel_launches": [],
    "a2ats_set_kernel_timing": [_I32],
    "a2ats_timed_kernels_ms": [_P],
}


def declared_symbols() -> list[str]:
    """Names of the functions include/a2ats.h declares."""
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"\b(a2ats_\w+)\s*\(", text)))


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m query_aware_vq_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        for name in ("a2ats_query_second_moment_workspace_size",
                     "a2ats_h_weighted_assign_workspace_size",
                     "a2ats_query_aware_assign_workspace_size",
                     "a2ats_select_retrieval_set_workspace_size",
                     "a2ats_rope_split_plain_assign_workspace_size",
                     "a2ats_code_attention_topk_workspace_size",
                     "a2ats_cholesky_rows_workspace_size",
                     "a2ats_kmeanspp_workspace_size",
                     "a2ats_subvector_assign_workspace_size",
                     "a2ats_subvector_query_aware_assign_workspace_size"):
            getattr(lib, name).restype = ctypes.c_size_t
        lib.a2ats_kernel_launches.restype = ctypes.c_uint64
        lib.a2ats_timed_kernels_ms.restype = ctypes.c_double
        lib.a2ats_status_string.restype = ctypes.c_char_p
        lib.a2ats_last_error.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def library():
    """The loaded ctypes handle of liba2ats.so."""
    return _load()


def kernel_launches() -> int:
    """Kernels the library has enqueued since it was loaded."""
    return int(_load().a2ats_kernel_launches())


def set_kernel_timing(enable: bool) -> None:
    """Record CUDA events around each stored-order tensor-core contraction."""
    _load().a2ats_set_kernel_timing(int(bool(enable)))


def timed_kernels_ms():
    """(summed milliseconds, number of timed launches) since the last call."""
    n = ctypes.c_int64(0)
    ms = _load().a2ats_timed_kernels_ms(ctypes.byref(n))
    return ms, n.value


def _check(fn: str, status: int):
    if status != 0:
        detail = _load().a2ats_last_error().decode() if status == -5 else ""
        raise A2ATSError(fn, status, detail)


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DTYPES[t.dtype]


def _dev(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous (the library reads and writes them "
                             "through their data pointers in row-major order)")
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device (the library has no CPU path)")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _as4(k: torch.Tensor) -> torch.Tensor:
    if k.dim() == 2:
        return k.view(1, 1, *k.shape)
    if k.dim() != 4:
        raise ValueError("keys must be [N, d] or [B, H, N, d]")
    return k


def _rope(rope):
    """None, a RopeParams, or a dict with window / far_offset / rope_base / interleaved."""
    if rope is None or isinstance(rope, RopeParams):
        return rope
    return RopeParams(int(rope["window"]), int(rope.get("far_offset", 0)),
                      float(rope.get("rope_base", 10000.0)), int(bool(rope.get("interleaved", 0))))


def _workspace(nbytes: int, device, ws, stream=None):
    """The caller's workspace, or a fresh one.  A fresh one is freed when the
    binding returns, while the call may still run on `stream`: recording the
    stream keeps the allocator from handing the memory out before then."""
    if ws is not None:
        return ws, ws.numel() * ws.element_size()
    ws = torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)
    if stream is not None:
        ws.record_stream(stream)
    return ws, int(nbytes)


def _lens(lengths):
    if lengths is not None and lengths.dtype != torch.int32:
        raise TypeError("lengths must be int32")
    return lengths


def a2ats_windowed_rope(k, *, window: int, far_offset: int = 0, rope_base: float = 10000.0,
                        interleaved: bool = False, lengths=None, out=None, out_dtype=None,
                        stream=None):
    """Windowed RoPE of every valid cached key against its sequence's decode
    position; returns `out` (same shape as k)."""
    _dev(k, lengths, out)
    k4 = _as4(k)
    if out is None:
        out = torch.empty(k.shape, dtype=out_dtype or k.dtype, device=k.device)
    o4 = _as4(out)
    p = RopeParams(int(window), int(far_offset), float(rope_base), int(bool(interleaved)))
    B, H, N, d = k4.shape
    _check("a2ats_windowed_rope", _load().a2ats_windowed_rope(
        _ptr(k4), _dt(k4), _ptr(o4), _dt(o4), B, H, N, d, _ptr(_lens(lengths)),
        ctypes.byref(p), _stream(stream)))
    return out


def a2ats_append_rows(cache, lengths, rows, *, stream=None):
    """Store rows [B, H, d] at position lengths[b] of every (b, h) of the
    cache [B, H, Ncap, d] and advance lengths (int32, device) by one."""
    _dev(cache, lengths, rows)
    if lengths is None or lengths.dtype != torch.int32:
        raise TypeError("lengths must be an int32 device tensor")
    if rows.dtype != cache.dtype:
        raise TypeError("rows and cache must share a dtype")
    B, H, N, d = cache.shape
    _check("a2ats_append_rows", _load().a2ats_append_rows(
        _ptr(cache), _dt(cache), B, H, N, d, _ptr(lengths), _ptr(rows), _stream(stream)))
    return cache


def a2ats_query_second_moment(queries, ridge: float = 1e-4, *, out=None, workspace=None,
                              stream=None):
    """H = (1/M) Q^T Q + ridge I per head; queries [H, M, d] (or [M, d])."""
    _dev(queries, out)
    q = queries if queries.dim() == 3 else queries.unsqueeze(0)
    Hh, M, d = q.shape
    if out is None:
        out = torch.empty((Hh, d, d), dtype=torch.float32, device=q.device)
    lib = _load()
    ws, nb = _workspace(lib.a2ats_query_second_moment_workspace_size(Hh, M, d), q.device,
                        workspace, stream)
    _check("a2ats_query_second_moment", lib.a2ats_query_second_moment(
        _ptr(q), _dt(q), Hh, M, d, float(ridge), _ptr(out), _ptr(ws), nb, _stream(stream)))
    return out if queries.dim() == 3 else out[0]


def a2ats_cholesky_factor(h, *, out=None, info=None, stream=None):
    """Lower-triangular L with H = L L^T per head; returns (L, info)."""
    _dev(h, out, info)
    h3 = h if h.dim() == 3 else h.unsqueeze(0)
    Hh, d, _ = h3.shape
    if out is None:
        out = torch.empty_like(h3, dtype=torch.float32)
    if info is None:
        info = torch.empty(Hh, dtype=torch.int32, device=h.device)
    _check("a2ats_cholesky_factor", _load().a2ats_cholesky_factor(
        _ptr(h3), Hh, d, _ptr(out), _ptr(info), _stream(stream)))
    return (out, info) if h.dim() == 3 else (out[0], info)


def _assign_common(x, codebook, codes):
    x4 = _as4(x)
    B, H, N, d = x4.shape
    cb = codebook if codebook.dim() == 3 else codebook.unsqueeze(0)
    if cb.dtype != x4.dtype:
        raise TypeError("codebook and keys must share a dtype")
    K = cb.shape[1]
    if codes is None:
        codes = torch.empty((B, H, N), dtype=torch.int32, device=x.device)
    return x4, cb, K, codes


def a2ats_h_weighted_assign(x, codebook, L=None, *, lengths=None, rope=None, rows="all",
                            perm=None, count=None, codes=None, workspace=None, stream=None,
                            reuse=False):
    """argmin_j |x~ L - c_j L|^2 per visited row (L None: plain VQ).
    reuse=True calls a2ats_h_weighted_assign_reuse: the codebook side is
    taken from `workspace` as the previous call with the same codebook, L,
    shapes, rope and rows left it."""
    _dev(x, codebook, L, lengths, perm, count, codes)
    x4, cb, K, codes = _assign_common(x, codebook, codes)
    B, H, N, d = x4.shape
    lib = _load()
    if reuse and workspace is None:
        raise ValueError("reuse needs the workspace of the preparing call")
    ws, nb = _workspace(lib.a2ats_h_weighted_assign_workspace_size(B, H, N, d, K), x.device,
                        workspace, stream)
    rp = _rope(rope)
    name = "a2ats_h_weighted_assign_reuse" if reuse else "a2ats_h_weighted_assign"
    _check(name, getattr(lib, name)(
        _ptr(x4), _dt(x4), B, H, N, d, _ptr(_lens(lengths)), _ptr(cb), K, _ptr(L),
        ctypes.byref(rp) if rp is not None else None, A2ATS_ROWS[rows], _ptr(perm), _ptr(count),
        _ptr(codes), _ptr(ws), nb, _stream(stream)))
    return codes


def a2ats_query_aware_assign(x, codebook, query=None, beta: float = 0.5, *, lengths=None,
                             rope=None, rows="all", perm=None, count=None, codes=None,
                             workspace=None, stream=None, reuse=False):
    """Cosine-blend assignment; query [B, H, d], or None for the proxy query
    (the key at the decode position after windowed RoPE).  reuse=True calls
    a2ats_query_aware_assign_reuse: the codebook side is the one the last
    call on `workspace` left (same codebook, shapes, beta = 1 or not, rope
    and rows), so a workspace must be given."""
    _dev(x, codebook, query, lengths, perm, count, codes)
    x4, cb, K, codes = _assign_common(x, codebook, codes)
    B, H, N, d = x4.shape
    if query is not None and query.dtype != x4.dtype:
        raise TypeError("query and keys must share a dtype")
    lib = _load()
    ws, nb = _workspace(lib.a2ats_query_aware_assign_workspace_size(B, H, N, d, K), x.device,
                        workspace, stream)
    rp = _rope(rope)
    if reuse and workspace is None:
        raise ValueError("reuse=True needs the workspace the codebook side was built in")
    name = "a2ats_query_aware_assign_reuse" if reuse else "a2ats_query_aware_assign"
    _check(name, getattr(lib, name)(
        _ptr(x4), _dt(x4), B, H, N, d, _ptr(_lens(lengths)), _ptr(cb), K, _ptr(query),
        float(beta), ctypes.byref(rp) if rp is not None else None, A2ATS_ROWS[rows], _ptr(perm),
        _ptr(count), _ptr(codes), _ptr(ws), nb, _stream(stream)))
    return codes


def a2ats_select_retrieval_set(keys, query=None, fraction: float = 0.2, *, lengths=None,
                               rope=None, perm=None, count=None, workspace=None, stream=None):
    """Retrieval split; returns (perm [B, H, N] int32, count [B, H] int32).
    perm[..., :count] are the retrieval rows ascending, the rest the bulk."""
    _dev(keys, query, lengths, perm, count)
    k4 = _as4(keys)
    B, H, N, d = k4.shape
    if query is not None and query.dtype != k4.dtype:
        raise TypeError("query and keys must share a dtype")
    if perm is None:
        perm = torch.empty((B, H, N), dtype=torch.int32, device=keys.device)
    if count is None:
        count = torch.empty((B, H), dtype=torch.int32, device=keys.device)
    lib = _load()
    ws, nb = _workspace(lib.a2ats_select_retrieval_set_workspace_size(B, H, N, d), keys.device,
                        workspace, stream)
    rp = _rope(rope)
    _check("a2ats_select_retrieval_set", lib.a2ats_select_retrieval_set(
        _ptr(k4), _dt(k4), B, H, N, d, _ptr(_lens(lengths)), _ptr(query), float(fraction),
        ctypes.byref(rp) if rp is not None else None, _ptr(perm), _ptr(count), _ptr(ws), nb,
        _stream(stream)))
    return perm, count


def a2ats_select_retrieval_set_rotated(keys, query=None, fraction: float = 0.2, *, rope,
                                       lengths=None, out=None, out_dtype=None, perm=None,
                                       count=None, workspace=None, stream=None):
    """Windowed RoPE of the cache and the retrieval split in one pass over
    the pre-RoPE keys; returns (out, perm, count), each exactly what
    a2ats_windowed_rope and a2ats_select_retrieval_set(rope=rope) return."""
    _dev(keys, query, lengths, out, perm, count)
    k4 = _as4(keys)
    B, H, N, d = k4.shape
    if query is not None and query.dtype != k4.dtype:
        raise TypeError("query and keys must share a dtype")
    if out is None:
        out = torch.empty(keys.shape, dtype=out_dtype or keys.dtype, device=keys.device)
    o4 = _as4(out)
    if perm is None:
        perm = torch.empty((B, H, N), dtype=torch.int32, device=keys.device)
    if count is None:
        count = torch.empty((B, H), dtype=torch.int32, device=keys.device)
    lib = _load()
    ws, nb = _workspace(lib.a2ats_select_retrieval_set_workspace_size(B, H, N, d), keys.device,
                        workspace, stream)
    rp = _rope(rope)
    _check("a2ats_select_retrieval_set_rotated", lib.a2ats_select_retrieval_set_rotated(
        _ptr(k4), _dt(k4), B, H, N, d, _ptr(_lens(lengths)), _ptr(query), float(fraction),
        ctypes.byref(rp), _ptr(o4), _dt(o4), _ptr(perm), _ptr(count), _ptr(ws), nb,
        _stream(stream)))
    return out, perm, count


def a2ats_rope_split_plain_assign(keys, codebook, query=None, fraction: float = 0.2, *, rope,
                                  lengths=None, out=None, perm=None, count=None, codes=None,
                                  reuse=False, split_done=None, split_stream=None, workspace=None,
                                  stream=None):
    """Windowed RoPE, the retrieval split and plain VQ of every row in one
    call over the pre-RoPE keys; returns (out, perm, count, codes).
    split_done: a torch.cuda.Event, recorded on the stream once out, perm and
    count are written (the codes follow).  split_stream: a torch.cuda.Stream
    (with split_done) that runs the split beside the rest of the call.
    reuse=True takes the codebook side from `workspace` as the previous call
    on it left it."""
    _dev(keys, codebook, query, lengths, out, perm, count, codes)
    k4, cb, K, codes = _assign_common(keys, codebook, codes)
    B, H, N, d = k4.shape
    if query is not None and query.dtype != k4.dtype:
        raise TypeError("query and keys must share a dtype")
    if out is None:
        out = torch.empty(keys.shape, dtype=keys.dtype, device=keys.device)
    if out.dtype != keys.dtype:
        raise TypeError("out must have the keys' dtype")
    o4 = _as4(out)
    if perm is None:
        perm = torch.empty((B, H, N), dtype=torch.int32, device=keys.device)
    if count is None:
        count = torch.empty((B, H), dtype=torch.int32, device=keys.device)
    lib = _load()
    if reuse and workspace is None:
        raise ValueError("reuse needs the workspace of the preparing call")
    ws, nb = _workspace(lib.a2ats_rope_split_plain_assign_workspace_size(B, H, N, d, K),
                        keys.device, workspace, stream)
    ev = None
    if split_done is not None:
        ev = split_done.cuda_event
        if not ev:
            raise ValueError("split_done must have been recorded once (its handle is made "
                             "lazily)")
    rp = _rope(rope)
    _check("a2ats_rope_split_plain_assign", lib.a2ats_rope_split_plain_assign(
        _ptr(k4), _dt(k4), B, H, N, d, _ptr(_lens(lengths)), _ptr(query), float(fraction),
        ctypes.byref(rp), _ptr(cb), K, _ptr(o4), _ptr(perm), _ptr(count), _ptr(codes),
        int(bool(reuse)), ev, _stream(split_stream) if split_stream is not None else None,
        _ptr(ws), nb, _stream(stream)))
    return out, perm, count, codes


def a2ats_code_attention_topk(keys, codes, codebook, query, fraction: float = 0.2, *, rope,
                              far_b: int = 2048, lengths=None, scores=None, perm=None,
                              count=None, workspace=None, stream=None):
    """Attention scores of the decode query with every cached key (far keys
    through their codes, window keys exactly) and the top tokens by them;
    returns (scores [B, H, N] fp32, perm, count)."""
    _dev(keys, codes, codebook, query, lengths, scores, perm, count)
    k4 = _as4(keys)
    B, H, N, d = k4.shape
    cb = codebook if codebook.dim() == 3 else codebook.unsqueeze(0)
    if cb.dtype != k4.dtype or query.dtype != k4.dtype:
        raise TypeError("keys, codebook and query must share a dtype")
    if codes.dtype != torch.int32:
        raise TypeError("codes must be int32")
    K = cb.shape[1]
    if scores is None:
        scores = torch.empty((B, H, N), dtype=torch.float32, device=keys.device)
    if perm is None:
        perm = torch.empty((B, H, N), dtype=torch.int32, device=keys.device)
    if count is None:
        count = torch.empty((B, H), dtype=torch.int32, device=keys.device)
    lib = _load()
    ws, nb = _workspace(lib.a2ats_code_attention_topk_workspace_size(B, H, N, d, K),
                        keys.device, workspace, stream)
    rp = _rope(rope)
    _check("a2ats_code_attention_topk", lib.a2ats_code_attention_topk(
        _ptr(k4), _dt(k4), B, H, N, d, _ptr(_lens(lengths)), _ptr(codes), _ptr(cb), K,
        _ptr(query), ctypes.byref(rp), int(far_b), float(fraction), _ptr(scores), _ptr(perm),
        _ptr(count), _ptr(ws), nb, _stream(stream)))
    return scores, perm, count


class CacheBytes(ctypes.Structure):
    """a2ats_cache_bytes: the byte accounting of a cache's keys and values
    as codes."""
    _fields_ = [("compressed_key_bytes", ctypes.c_double),
                ("compressed_value_bytes", ctypes.c_double),
                ("fp16_key_bytes", ctypes.c_double), ("fp16_value_bytes", ctypes.c_double),
                ("compression_ratio", ctypes.c_double), ("codebook_bytes", ctypes.c_double),
                ("assigned_avg_bits", ctypes.c_double)]


def a2ats_byte_accounting(tokens: int, d: int, sub_dim: int, codebook_bits: int) -> dict:
    """The page's byte accounting of `tokens` keys and values of width d
    (host arithmetic through the C ABI)."""
    out = CacheBytes()
    _check("a2ats_byte_accounting", _load().a2ats_byte_accounting(
        int(tokens), int(d), int(sub_dim), int(codebook_bits), ctypes.byref(out)))
    return {name: getattr(out, name) for name, _ in CacheBytes._fields_}


def a2ats_dequantize(codes, codebook, *, lengths=None, out=None, stream=None):
    """Keys reconstructed from their codes: out[b, h, j] = codebook[h,
    codes[b, h, j]] for rows j < len[b]; returns out [B, H, N, d]."""
    _dev(codes, codebook, lengths, out)
    if codes.dtype != torch.int32 or codes.dim() != 3:
        raise TypeError("codes must be int32 [B, H, N]")
    cb = codebook if codebook.dim() == 3 else codebook.unsqueeze(0)
    B, H, N = codes.shape
    K, d = cb.shape[1], cb.shape[2]
    if out is None:
        out = torch.empty((B, H, N, d), dtype=cb.dtype, device=codes.device)
    _check("a2ats_dequantize", _load().a2ats_dequantize(
        _ptr(codes), _ptr(cb), _dt(cb), B, H, N, d, K, _ptr(_lens(lengths)), _ptr(out),
        _stream(stream)))
    return out


def a2ats_copy_retrieval_rows(src, dst, perm, count, *, lengths=None, stream=None):
    """dst[b, h, j] = src[b, h, j] on the retrieval rows of the split;
    returns dst (int32 [B, H, N] device tensors)."""
    _dev(src, dst, perm, count, lengths)
    if src.dtype != torch.int32 or dst.dtype != torch.int32 or src.shape != dst.shape:
        raise TypeError("src and dst must be int32 tensors of one shape")
    B, H, N = dst.shape
    _check("a2ats_copy_retrieval_rows", _load().a2ats_copy_retrieval_rows(
        _ptr(src), _ptr(dst), B, H, N, _ptr(_lens(lengths)), _ptr(perm), _ptr(count),
        _stream(stream)))
    return dst


def a2ats_subvector_assign(x, codebook, sub_dim: int, L=None, *, lengths=None, perm=None,
                           count=None, codes=None, workspace=None, stream=None):
    """Sub-vector codes [B, H, N, d // sub_dim] of x [B, H, N, d] against
    the per-head tables codebook [H, K, sub_dim] (x's dtype): the H-weighted
    rule with L [H, sub_dim, sub_dim] on the retrieval tokens of the split
    (perm, count; every token when they are None), plain VQ elsewhere (and
    everywhere when L is None)."""
    _dev(x, codebook, L, lengths, perm, count, codes)
    x4 = _as4(x)
    B, H, N, d = x4.shape
    cb = codebook if codebook.dim() == 3 else codebook.unsqueeze(0)
    if cb.dtype != x4.dtype or cb.shape[2] != sub_dim:
        raise TypeError("codebook must be [H, K, sub_dim] in the dtype of x")
    K = cb.shape[1]
    if codes is None:
        codes = torch.empty((B, H, N, d // sub_dim), dtype=torch.int32, device=x.device)
    lib = _load()
    ws, nb = _workspace(lib.a2ats_subvector_assign_workspace_size(B, H, N, d, sub_dim, K),
                        x.device, workspace, stream)
    _check("a2ats_subvector_assign", lib.a2ats_subvector_assign(
        _ptr(x4), _dt(x4), B, H, N, d, _ptr(_lens(lengths)), int(sub_dim), _ptr(cb), K,
        _ptr(L), _ptr(perm), _ptr(count), _ptr(codes), _ptr(ws), nb, _stream(stream)))
    return codes


def a2ats_subvector_query_aware_assign(x, codebook, sub_dim: int, query=None,
                                       beta: float = 0.5, *, lengths=None, perm=None,
                                       count=None, codes=None, workspace=None, stream=None):
    """Sub-vector codes [B, H, N, d // sub_dim] of x [B, H, N, d]: the cosine
    blend with the query's slice on the retrieval tokens of the split (perm,
    count; every token when they are None), plain VQ elsewhere.  query [B,
    H, d] in x's dtype, or None for the row of x at t = len - 1."""
    _dev(x, codebook, query, lengths, perm, count, codes)
    x4 = _as4(x)
    B, H, N, d = x4.shape
    cb = codebook if codebook.dim() == 3 else codebook.unsqueeze(0)
    if cb.dtype != x4.dtype or cb.shape[2] != sub_dim:
        raise TypeError("codebook must be [H, K, sub_dim] in the dtype of x")
    if query is not None and query.dtype != x4.dtype:
        raise TypeError("query must share the dtype of x")
    K = cb.shape[1]
    if codes is None:
        codes = torch.empty((B, H, N, d // sub_dim), dtype=torch.int32, device=x.device)
    lib = _load()
    ws, nb = _workspace(
        lib.a2ats_subvector_query_aware_assign_workspace_size(B, H, N, d, sub_dim, K), x.device,
        workspace, stream)
    _check("a2ats_subvector_query_aware_assign", lib.a2ats_subvector_query_aware_assign(
        _ptr(x4), _dt(x4), B, H, N, d, _ptr(_lens(lengths)), int(sub_dim), _ptr(cb), K,
        _ptr(query), float(beta), _ptr(perm), _ptr(count), _ptr(codes), _ptr(ws), nb,
        _stream(stream)))
    return codes


def _as3(t: torch.Tensor, what: str) -> torch.Tensor:
    if t.dim() == 2:
        return t.unsqueeze(0)
    if t.dim() != 3:
        raise ValueError(f"{what} must be [n, d] or [H, n, d]")
    return t


def a2ats_cholesky_rows(x, L, *, out=None, workspace=None, stream=None):
    """z = x L per head: x [H, n, d] (or [n, d]) in any supported dtype, L
    [H, d, d] fp32 (lower triangle read); returns fp32 z of x's shape."""
    _dev(x, L, out)
    x3 = _as3(x, "x")
    L3 = L if L.dim() == 3 else L.unsqueeze(0)
    Hh, n, d = x3.shape
    if L3.dtype != torch.float32 or L3.shape != (Hh, d, d):
        raise TypeError("L must be fp32 [H, d, d]")
    if out is None:
        out = torch.empty((Hh, n, d), dtype=torch.float32, device=x.device)
    lib = _load()
    ws, nb = _workspace(lib.a2ats_cholesky_rows_workspace_size(Hh, n, d), x.device, workspace,
                        stream)
    _check("a2ats_cholesky_rows", lib.a2ats_cholesky_rows(
        _ptr(x3), _dt(x3), Hh, n, d, _ptr(L3), _ptr(out), _ptr(ws), nb, _stream(stream)))
    return out if x.dim() == 3 else out[0]


def a2ats_cholesky_solve_rows(zc, L, *, out=None, stream=None):
    """c with c L = zc per head (z-space rows back to key space): zc [H, rows,
    d] fp32 (or [rows, d]), L [H, d, d] fp32 lower triangular."""
    _dev(zc, L, out)
    z3 = _as3(zc, "zc")
    L3 = L if L.dim() == 3 else L.unsqueeze(0)
    Hh, rows, d = z3.shape
    if z3.dtype != torch.float32 or L3.dtype != torch.float32 or L3.shape != (Hh, d, d):
        raise TypeError("zc must be fp32 [H, rows, d] and L fp32 [H, d, d]")
    if out is None:
        out = torch.empty((Hh, rows, d), dtype=torch.float32, device=zc.device)
    _check("a2ats_cholesky_solve_rows", _load().a2ats_cholesky_solve_rows(
        _ptr(z3), Hh, rows, d, _ptr(L3), _ptr(out), _stream(stream)))
    return out if zc.dim() == 3 else out[0]


def a2ats_kmeanspp(z, K: int, u, iters: int, *, centroids=None, codes=None, objective=None,
                   workspace=None, stream=None):
    """k-means++ seeding with the uniform draws u [H, K] (fp64), then `iters`
    Lloyd rounds, on fp32 rows z [H, n, d] (or [n, d] with u [K]).  Returns
    (centroids [H, K, d] fp32, codes [H, n] int32, objective [H, iters + 1]
    fp64), without the head axis for 2-d z."""
    _dev(z, u, centroids, codes, objective)
    z3 = _as3(z, "z")
    Hh, n, d = z3.shape
    u2 = (u if u.dim() == 2 else u.unsqueeze(0)).contiguous()
    if z3.dtype != torch.float32 or u2.dtype != torch.float64 or u2.shape != (Hh, K):
        raise TypeError("z must be fp32 [H, n, d] and u fp64 [H, K]")
    dev = z.device
    if centroids is None:
        centroids = torch.empty((Hh, K, d), dtype=torch.float32, device=dev)
    if codes is None:
        codes = torch.empty((Hh, n), dtype=torch.int32, device=dev)
    if objective is None:
        objective = torch.empty((Hh, iters + 1), dtype=torch.float64, device=dev)
    lib = _load()
    ws, nb = _workspace(lib.a2ats_kmeanspp_workspace_size(Hh, n, d, K), dev, workspace, stream)
    _check("a2ats_kmeanspp", lib.a2ats_kmeanspp(
        _ptr(z3), Hh, n, d, int(K), _ptr(u2), int(iters), _ptr(centroids),
        _ptr(codes), _ptr(objective), _ptr(ws), nb, _stream(stream)))
    if z.dim() == 3:
        return centroids, codes, objective
    return centroids[0], codes[0], objective[0]


def split_views(perm, count, b: int = 0, h: int = 0, n: int | None = None):
    """(retrieval_idx, bulk_idx) of one (b, h), as the API page returns them."""
    c = int(count[b, h])
    p = perm[b, h] if n is None else perm[b, h, :n]
    return p[:c], p[c:]
