"""Seeded synthetic inputs shaped like the workloads of the A2ATS pages.

This module only draws random numbers and casts them to the storage dtype.
It holds none of the method's arithmetic (no RoPE, no second moment, no
Cholesky, no distances), so both the CPU oracle and the CUDA path can take
their inputs from it without sharing any part of the computation.

The pages run Llama-class models (Llama-3.2-3B, head_dim 128; the calibration
snippet on the A2ATS docs page collects keys shaped [4096, 8, 128]).  No
model, dataset or weights exist here, so every tensor is drawn from the
recipes below with numpy's PCG64 generator:

* correlated Gaussian keys: ``k = g A_h^T / sqrt(d)`` with ``A_h`` i.i.d.
  N(0, 1) (seed ``h``) and ``g ~ N(0, I)``; four channels of ``A_h``'s
  choosing are multiplied by 8 (outlier channels);
* queries: ``q = g1 A_h^T / sqrt(d) + sqrt(0.5) g2`` (no outlier channels);
* codebooks: ``K`` rows drawn without replacement from a separate sample of
  ``4K`` keys of the same head;
* heavy-tailed keys (wide-head stress): Student-t (nu=3) times a per-channel
  scale that is log-uniform in [0.1, 10];
* ill-conditioned H (wide-head stress): ``Q diag(lambda) Q^T + ridge I``, Q
  from the QR factorisation of a Gaussian matrix with signs fixed so R has a
  positive diagonal, lambda log-uniform in [1e-3, 1e3].

Casts to bf16 / fp16 go through torch (round to nearest even).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass(frozen=True)
class Workload:
    """Sizes and knobs of one synthetic workload (names follow the pages)."""

    name: str
    B: int                  # sequences
    H: int                  # KV heads
    N: int                  # cached keys per (b, h) (capacity for decode)
    d: int                  # head_dim = VQ width
    dtype: str              # storage dtype of keys / queries / codebooks
    K: int                  # centroids per head
    W: int                  # trailing exact-RoPE window
    fraction: float         # retrieval_fraction
    rope_base: float
    M: int = 0              # calibration queries per head (0: H is given)
    ridge: float = 1e-4
    betas: tuple = (1.0,)
    far_offset: int = 0
    keys: str = "gaussian"  # or "student_t"
    h_given: bool = False   # H drawn directly (ill-conditioned) instead of from queries
    decode_steps: int = 0
    calibrate_in_step: bool = False  # H and L recomputed by every step (else once, ahead)
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    # one head, fp32, small enough for every oracle routine in seconds
    "tiny": Workload("tiny", B=1, H=1, N=1024, d=128, dtype="f32", K=256, W=64,
                     fraction=0.1, rope_base=500000.0, M=512, betas=(1.0, 0.5)),
    # one attention layer of a Llama-3.2-3B-shaped model
    "llama32_3b_layer": Workload("llama32_3b_layer", B=1, H=8, N=32768, d=128, dtype="bf16",
                                 K=1024, W=512, fraction=0.05, rope_base=500000.0, M=8192),
    # Llama-3-8B-shaped long context, batch 4
    "llama3_8b_long": Workload("llama3_8b_long", B=4, H=8, N=131072, d=128, dtype="bf16",
                               K=4096, W=1024, fraction=0.02, rope_base=500000.0, M=65536,
                               calibrate_in_step=True),
    # decode streaming: 64 sequences, lengths U[8192, 32768], one new key per
    # (sequence, head) per step, 128 steps
    "decode_stream": Workload("decode_stream", B=64, H=8, N=32768 + 128, d=128, dtype="bf16",
                              K=1024, W=256, fraction=0.1, rope_base=500000.0, betas=(0.7,),
                              decode_steps=128),
    # wide heads, heavy tails, ill-conditioned H
    "wide_head": Workload("wide_head", B=1, H=32, N=65536, d=256, dtype="f16", K=8192, W=2048,
                          fraction=0.1, rope_base=10000.0, keys="student_t", h_given=True),
}


def _outliers_and_mixing(h: int, d: int):
    rng = np.random.default_rng(h)
    A = rng.standard_normal((d, d))
    out = rng.choice(d, 4, replace=False)
    return A, out


def _gauss_keys(rng, A, out, n, d, chunk=1 << 16):
    res = np.empty((n, d), dtype=np.float32)
    At = (A.T / math.sqrt(d)).astype(np.float64)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        g = rng.standard_normal((e - s, d))
        k = g @ At
        k[:, out] *= 8.0
        res[s:e] = k
    return res


def _channel_scale(h: int, d: int):
    rng = np.random.default_rng(7000 + h)
    return np.exp(rng.uniform(math.log(0.1), math.log(10.0), size=d))


def _t_keys(rng, scale, n, d, chunk=1 << 16):
    res = np.empty((n, d), dtype=np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        res[s:e] = rng.standard_t(3.0, size=(e - s, d)) * scale
    return res


def _keys_for(w: Workload, b: int, h: int, n: int) -> np.ndarray:
    rng = np.random.default_rng(1000 + b * w.H + h)
    if w.keys == "student_t":
        return _t_keys(rng, _channel_scale(h, w.d), n, w.d)
    A, out = _outliers_and_mixing(h, w.d)
    return _gauss_keys(rng, A, out, n, w.d)


def _to_storage(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "f16":
        # heavy-tailed draws can exceed the fp16 range; clamp to the largest
        # finite value so every stored key is finite
        t = t.clamp_(-65504.0, 65504.0)
    return t.to(DTYPES[dtype])


def keys(w: Workload, rows: int | None = None, threads: int = 8,
         batch_offset: int = 0) -> torch.Tensor:
    """Keys [B, H, rows, d] in the storage dtype (rows defaults to N).
    batch_offset: the batch holds sequences batch_offset .. batch_offset + B - 1
    of the stream (another batch of the same workload)."""
    n = w.N if rows is None else rows
    out = torch.empty((w.B, w.H, n, w.d), dtype=DTYPES[w.dtype])

    def one(bh):
        b, h = divmod(bh, w.H)
        out[b, h] = _to_storage(_keys_for(w, b + batch_offset, h, n), w.dtype)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, range(w.B * w.H)))
    return out


def head_keys(w: Workload, b: int, h: int, rows: int | None = None) -> torch.Tensor:
    """Keys [1, 1, rows, d] of sequence b and head h alone, the same values
    keys(w)[b, h] holds."""
    n = w.N if rows is None else rows
    return _to_storage(_keys_for(w, b, h, n), w.dtype).view(1, 1, n, w.d)


def queries(w: Workload, M: int | None = None) -> torch.Tensor:
    """Calibration queries [H, M, d] in the storage dtype."""
    M = w.M if M is None else M
    out = torch.empty((w.H, M, w.d), dtype=DTYPES[w.dtype])
    for h in range(w.H):
        A, _ = _outliers_and_mixing(h, w.d)
        rng = np.random.default_rng(2000 + h)
        q = rng.standard_normal((M, w.d)) @ (A.T / math.sqrt(w.d))
        q += math.sqrt(0.5) * rng.standard_normal((M, w.d))
        out[h] = _to_storage(q, w.dtype)
    return out


def codebook(w: Workload, K: int | None = None) -> torch.Tensor:
    """Codebooks [H, K, d]: K rows sampled without replacement from a separate
    draw of 4K keys of the same head."""
    K = w.K if K is None else K
    out = torch.empty((w.H, K, w.d), dtype=DTYPES[w.dtype])
    for h in range(w.H):
        rng = np.random.default_rng(3000 + h)
        if w.keys == "student_t":
            src = _t_keys(rng, _channel_scale(h, w.d), 4 * K, w.d)
        else:
            A, o = _outliers_and_mixing(h, w.d)
            src = _gauss_keys(rng, A, o, 4 * K, w.d)
        idx = rng.choice(4 * K, K, replace=False)
        out[h] = _to_storage(src[idx], w.dtype)
    return out


def given_h(w: Workload) -> torch.Tensor:
    """Ill-conditioned second-moment matrices [H, d, d] fp32 (wide-head stress)."""
    out = torch.empty((w.H, w.d, w.d), dtype=torch.float32)
    for h in range(w.H):
        rng = np.random.default_rng(4000 + h)
        G = rng.standard_normal((w.d, w.d))
        Q, R = np.linalg.qr(G)
        Q = Q * np.sign(np.diag(R))[None, :]
        lam = np.exp(rng.uniform(math.log(1e-3), math.log(1e3), size=w.d))
        Hm = (Q * lam[None, :]) @ Q.T + w.ridge * np.eye(w.d)
        Hm = 0.5 * (Hm + Hm.T)
        out[h] = torch.from_numpy(Hm.astype(np.float32))
    return out


def decode_lengths(w: Workload) -> np.ndarray:
    """Initial context lengths of the decode workload, U[8192, 32768]."""
    rng = np.random.default_rng(6000)
    return rng.integers(8192, 32768, size=w.B, endpoint=True).astype(np.int32)


def decode_new_keys(w: Workload, step: int) -> torch.Tensor:
    """The keys appended at one decode step, [B, H, d]."""
    rng = np.random.default_rng(5000 + step)
    out = np.empty((w.B, w.H, w.d), dtype=np.float32)
    for h in range(w.H):
        A, o = _outliers_and_mixing(h, w.d)
        out[:, h] = _gauss_keys(rng, A, o, w.B, w.d)
    return _to_storage(out, w.dtype)


def gaussian(shape, seed: int, dtype: str = "f32", scale: float = 1.0) -> torch.Tensor:
    """Plain i.i.d. N(0, scale^2) tensor in the given storage dtype."""
    rng = np.random.default_rng(seed)
    return _to_storage(rng.standard_normal(shape) * scale, dtype)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some sizes changed (for small parity cases)."""
    from dataclasses import replace
    return replace(w, **changes)
