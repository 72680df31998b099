"""fp64 CPU oracle of the A2ATS hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import this module.  The product path (the CUDA library and its Python
binding) never imports, links or runs anything here, and this module never
imports the product.  Inputs come from the seeded generators in ``synth``.

Every routine decodes its inputs to fp64 exactly (bf16 / fp16 / fp32 are
subsets of fp64) and calls the plain C implementation in ``a2ats_oracle.c``.
The C file cites, routine by routine, the page section it follows.

``pipeline_step`` composes the routines the way the pages' cache wrapper
composes them for one step (v0.39.0 page, "How it works"; deploy-preview page,
"Per-step re-rotation"), under the readings listed with it.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import sys
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "a2ats_oracle.c")
_LIB = os.path.join(_HERE, "liba2ats_oracle.so")

_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)


def compile_source(src: str, out: str) -> str:
    """gcc the C source `src` (which includes a2ats_oracle.h from this
    directory) into the shared library `out`, with no FMA contraction so
    results do not depend on the host ISA."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", "-I", _HERE, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle (compile_source) unless the library is current."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "a2ats_oracle.h"))):
        tmp = _LIB + f".tmp{os.getpid()}"
        compile_source(_SRC, tmp)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        # A2ATS_ORACLE_LIB: a library built from a planted-mistake copy of the
        # source, for the tests that check the pins catch such mistakes
        lib = ctypes.CDLL(os.environ.get("A2ATS_ORACLE_LIB") or build())
        lib.orc_rope_row.argtypes = [_f64p, _f64p, ctypes.c_int64, ctypes.c_double,
                                     ctypes.c_double, ctypes.c_int]
        lib.orc_windowed_rope.argtypes = [_f64p, _f64p, ctypes.c_int64, ctypes.c_int64, _i64p,
                                          _i64p, ctypes.c_int64, ctypes.c_double,
                                          ctypes.c_double, ctypes.c_int]
        lib.orc_query_second_moment.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_double, _f64p]
        lib.orc_cholesky.argtypes = [_f64p, ctypes.c_int64, _f64p]
        lib.orc_cholesky.restype = ctypes.c_int
        for fn in (lib.orc_assign_quadratic, lib.orc_assign_cholesky):
            fn.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64, _f64p, ctypes.c_int64,
                           _f64p, _i32p, _f64p, _f64p, ctypes.c_int]
        lib.orc_assign_blend.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64, _f64p,
                                         ctypes.c_int64, _f64p, ctypes.c_int64,
                                         ctypes.c_double, _i32p, _f64p, _f64p, ctypes.c_int]
        lib.orc_select_retrieval_set.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64, _f64p,
                                                 ctypes.c_double, _i32p, _f64p, _f64p]
        lib.orc_select_retrieval_set.restype = ctypes.c_int64
        lib.orc_code_attention_topk.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_int64, _i32p, _f64p, ctypes.c_int64,
                                                _f64p, ctypes.c_int64, ctypes.c_double,
                                                ctypes.c_double, ctypes.c_int, ctypes.c_double,
                                                _i32p, _f64p, _f64p]
        lib.orc_code_attention_topk.restype = ctypes.c_int64
        for fn in (lib.orc_cholesky_rows, lib.orc_cholesky_solve_rows):
            fn.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64, _f64p, _f64p]
        lib.orc_dequantize.argtypes = [_i32p, ctypes.c_int64, _f64p, ctypes.c_int64,
                                       ctypes.c_int64, _f64p]
        lib.orc_kmeanspp.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                     _f64p, ctypes.c_int64, _f64p, _i32p, _f64p]
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    """Exact fp64 copy of a numpy array or torch tensor (bf16 included)."""
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        import torch
        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a, t):
    return a.ctypes.data_as(t)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------- #
# single routines
# --------------------------------------------------------------------------- #
def rope_row(x, pos: float, base: float, interleaved: bool = False) -> np.ndarray:
    x = _f64(x)
    y = np.empty_like(x)
    _load().orc_rope_row(_p(x, _f64p), _p(y, _f64p), x.shape[-1], float(pos), float(base),
                         int(interleaved))
    return y


def windowed_rope(x, p, t, window: int, far_offset: float, base: float,
                  interleaved: bool = False) -> np.ndarray:
    """x [rows, d]; p, t [rows] positions and decode positions."""
    x = _f64(x).reshape(-1, np.shape(x)[-1])
    rows, d = x.shape
    p = np.ascontiguousarray(np.broadcast_to(np.asarray(p, dtype=np.int64), (rows,)))
    t = np.ascontiguousarray(np.broadcast_to(np.asarray(t, dtype=np.int64), (rows,)))
    y = np.empty_like(x)
    _load().orc_windowed_rope(_p(x, _f64p), _p(y, _f64p), rows, d, _p(p, _i64p), _p(t, _i64p),
                              int(window), float(far_offset), float(base), int(interleaved))
    return y


def query_second_moment(q, ridge: float) -> np.ndarray:
    q = _f64(q)
    M, d = q.shape
    h = np.empty((d, d))
    _load().orc_query_second_moment(_p(q, _f64p), M, d, float(ridge), _p(h, _f64p))
    return h


def cholesky(h):
    """Returns (L, info): info = 0, or the 1-based order of the first leading
    minor that is not positive definite."""
    h = _f64(h)
    d = h.shape[0]
    l = np.empty((d, d))
    info = _load().orc_cholesky(_p(h, _f64p), d, _p(l, _f64p))
    return l, int(info)


def assign_quadratic(x, c, h, nthreads: int | None = None):
    x, c, h = _f64(x), _f64(c), _f64(h)
    n, d = x.shape
    K = c.shape[0]
    code = np.empty(n, np.int32)
    d1, d2 = np.empty(n), np.empty(n)
    _load().orc_assign_quadratic(_p(x, _f64p), n, d, _p(c, _f64p), K, _p(h, _f64p),
                                 _p(code, _i32p), _p(d1, _f64p), _p(d2, _f64p),
                                 nthreads or default_threads())
    return code, d1, d2


def assign_cholesky(x, c, l=None, nthreads: int | None = None):
    x, c = _f64(x), _f64(c)
    n, d = x.shape
    K = c.shape[0]
    lp = None
    if l is not None:
        l = _f64(l)
        lp = _p(l, _f64p)
    code = np.empty(n, np.int32)
    d1, d2 = np.empty(n), np.empty(n)
    _load().orc_assign_cholesky(_p(x, _f64p), n, d, _p(c, _f64p), K, lp, _p(code, _i32p),
                                _p(d1, _f64p), _p(d2, _f64p), nthreads or default_threads())
    return code, d1, d2


def assign_blend(x, c, q, beta: float, nthreads: int | None = None):
    """q: [d] shared query, or [n, d] one query per row."""
    x, c, q = _f64(x), _f64(c), _f64(q)
    n, d = x.shape
    K = c.shape[0]
    q_stride = d if q.ndim == 2 else 0
    code = np.empty(n, np.int32)
    s1, s2 = np.empty(n), np.empty(n)
    _load().orc_assign_blend(_p(x, _f64p), n, d, _p(c, _f64p), K, _p(q, _f64p), q_stride,
                             float(beta), _p(code, _i32p), _p(s1, _f64p), _p(s2, _f64p),
                             nthreads or default_threads())
    return code, s1, s2


def select_retrieval_set(keys, q, fraction: float):
    """Returns (perm, count, scores, kth_score)."""
    keys, q = _f64(keys), _f64(q)
    n, d = keys.shape
    perm = np.empty(n, np.int32)
    scores = np.empty(n)
    kth = np.empty(1)
    count = _load().orc_select_retrieval_set(_p(keys, _f64p), n, d, _p(q, _f64p),
                                             float(fraction), _p(perm, _i32p),
                                             _p(scores, _f64p), _p(kth, _f64p))
    return perm, int(count), scores, float(kth[0])


def code_attention_topk(keys, t: int, codes, codebook, q, window: int, far_b: float,
                        base: float, fraction: float, interleaved: bool = False):
    """Code-based attention scores of one (b, h) and its top tokens; keys
    [n, d] pre-RoPE, codes [n], codebook [K, d], q [d] pre-RoPE at position t.
    Returns (perm, count, scores, kth_score)."""
    keys, codebook, q = _f64(keys), _f64(codebook), _f64(q)
    n, d = keys.shape
    K = codebook.shape[0]
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    perm = np.empty(n, np.int32)
    scores = np.empty(n)
    kth = np.empty(1)
    count = _load().orc_code_attention_topk(
        _p(keys, _f64p), n, d, int(t), _p(codes, _i32p), _p(codebook, _f64p), K, _p(q, _f64p),
        int(window), float(far_b), float(base), int(bool(interleaved)), float(fraction),
        _p(perm, _i32p), _p(scores, _f64p), _p(kth, _f64p))
    return perm, int(count), scores, float(kth[0])


def dequantize(codes, codebook) -> np.ndarray:
    """codes [n] int32, codebook [K, d]: [n, d] of the codes' centroids
    (zeros for a code outside [0, K))."""
    codebook = _f64(codebook)
    K, d = codebook.shape
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    n = codes.shape[0]
    out = np.empty((n, d))
    _load().orc_dequantize(_p(codes, _i32p), n, _p(codebook, _f64p), K, d, _p(out, _f64p))
    return out


def cholesky_rows(x, l) -> np.ndarray:
    """z = x L for rows x [n, d] (the change of variables of the Cholesky
    route, API page, a2ats_cholesky_factor)."""
    x = _f64(x)
    l = _f64(l)
    n, d = x.shape
    assert l.shape == (d, d)
    z = np.empty((n, d))
    _load().orc_cholesky_rows(_p(x, _f64p), n, d, _p(l, _f64p), _p(z, _f64p))
    return z


def cholesky_solve_rows(z, l) -> np.ndarray:
    """c [n, d] with c L = z, L lower triangular (z-space centroids mapped
    back to key space)."""
    z = _f64(z)
    l = _f64(l)
    n, d = z.shape
    assert l.shape == (d, d)
    c = np.empty((n, d))
    _load().orc_cholesky_solve_rows(_p(z, _f64p), n, d, _p(l, _f64p), _p(c, _f64p))
    return c


def kmeanspp(z, K: int, u, iters: int):
    """k-means++ seeding with uniform draws u [K], then `iters` Lloyd rounds,
    on points z [n, d].  Returns (centroids [K, d], codes [n], objective
    [iters + 1])."""
    z = _f64(z)
    n, d = z.shape
    u = np.ascontiguousarray(u, dtype=np.float64)
    assert u.shape == (K,)
    cent = np.empty((K, d))
    codes = np.empty(n, np.int32)
    obj = np.empty(iters + 1)
    _load().orc_kmeanspp(_p(z, _f64p), n, d, K, _p(u, _f64p), int(iters), _p(cent, _f64p),
                         _p(codes, _i32p), _p(obj, _f64p))
    return cent, codes, obj


def byte_accounting(tokens: int, d: int, sub_dim: int, codebook_bits: int) -> dict:
    """The v0.39.0 page's byte accounting of a cache's keys and values
    ("Byte accounting"; "What you get with the defaults"): each key and each
    value of width d stores d / sub_dim codes of codebook_bits bits; fp16
    stores 16 bits per number; the ratio is the combined fp16 size over the
    combined compressed size; the codebook is one table of 2^bits entries of
    sub_dim fp16 numbers."""
    groups = d // sub_dim
    ck = tokens * groups * codebook_bits / 8.0
    fk = tokens * d * 2.0
    cv, fv = ck, fk
    ratio = (fk + fv) / (ck + cv) if ck + cv else 16.0 * sub_dim / codebook_bits
    return {"compressed_key_bytes": ck, "compressed_value_bytes": cv,
            "fp16_key_bytes": fk, "fp16_value_bytes": fv,
            "compression_ratio": ratio,
            "codebook_bytes": float((1 << codebook_bits) * sub_dim * 2),
            "assigned_avg_bits": codebook_bits / sub_dim}


def retrieval_count(fraction: float, n: int) -> int:
    """ceil(fraction * n) as the API page states it (IEEE double)."""
    return min(n, max(0, math.ceil(float(fraction) * n)))


# --------------------------------------------------------------------------- #
# one step of the path, composed
# --------------------------------------------------------------------------- #
@dataclass
class StepResult:
    k_tilde: np.ndarray       # [n, d] windowed-RoPE keys (fp64)
    perm: np.ndarray          # [n] retrieval indices ascending, then bulk ascending
    count: int
    scores: np.ndarray        # [n] key-query cosine
    kth: float                # smallest retained score
    codes: np.ndarray         # [n] centroid index per key
    gap: np.ndarray           # [n] relative top-2 gap of the rule that chose the code


def pipeline_step(k, t: int, codebook, window: int, far_offset: int, base: float,
                  fraction: float, l=None, beta: float = 1.0, interleaved: bool = False,
                  nthreads: int | None = None) -> StepResult:
    """One step for one (sequence, head): windowed RoPE of every cached key
    against decode position t -> retrieval split with the proxy query (the key
    at t after windowed RoPE) -> retrieval rows assigned by the H-weighted rule
    when L is given, else by the cosine blend with that query; bulk rows by
    plain nearest-centroid VQ.  k: [n, d] with n = t + 1 cached keys."""
    k = _f64(k)
    n, d = k.shape
    pos = np.arange(n, dtype=np.int64)
    kt = windowed_rope(k, pos, t, window, far_offset, base, interleaved)
    q = kt[t]
    perm, count, scores, kth = select_retrieval_set(kt, q, fraction)
    codes = np.empty(n, np.int32)
    gap = np.empty(n)
    ret, bulk = perm[:count], perm[count:]
    c = _f64(codebook)
    if count:
        if l is not None:
            cr, a, b = assign_cholesky(kt[ret], c, l, nthreads)
            g = (b - a) / np.where(b > 0, b, 1.0)
        else:
            cr, a, b = assign_blend(kt[ret], c, q, beta, nthreads)
            g = (b - a) / np.where(b > 0, b, 1.0) if beta == 1.0 else (a - b)
        codes[ret], gap[ret] = cr, g
    if n - count:
        cb, a, b = assign_cholesky(kt[bulk], c, None, nthreads)
        codes[bulk], gap[bulk] = cb, (b - a) / np.where(b > 0, b, 1.0)
    return StepResult(kt, perm, count, scores, kth, codes, gap)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
