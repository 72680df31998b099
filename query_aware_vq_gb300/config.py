"""The cache settings of the v0.39.0 page's A2ATS configuration, with its
defaults and its checks (configuration reference and troubleshooting list):
head_dim even and a multiple of a2ats_sub_dim, beta and retrieval_fraction
in [0, 1], query_h sub_dim x sub_dim, a codebook of 2^bits entries of
sub_dim numbers.  `validate()` raises ValueError on the first violated
rule; the same ranges are enforced again by the C ABI calls the settings
reach.  `subvector_step()` builds the sub-vector step these settings
describe, `factor()` the Cholesky factor of query_h it takes, and
`byte_accounting()` is the page's storage arithmetic for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Any


@dataclass
class A2ATSConfig:
    head_dim: int
    window: int = 128
    sub_dim: int = 8
    codebook_bits: int = 8
    use_query_aware: bool = True
    query_h: Any = None        # [sub_dim, sub_dim] (or [H, sub_dim, sub_dim]) second moment
    beta: float = 0.5          # blend weight, used when query_h is absent
    retrieval_fraction: float = 0.20
    b: int = 2048              # far relative position carried by the query
    rope_base: float = 10000.0
    codebook: Any = None       # [2^bits, sub_dim] or [H, 2^bits, sub_dim]

    @property
    def n_centroids(self) -> int:
        return 1 << self.codebook_bits

    def validate(self) -> "A2ATSConfig":
        if not isinstance(self.head_dim, int) or self.head_dim <= 0 or self.head_dim % 2:
            raise ValueError(f"head_dim must be a positive even integer, got {self.head_dim!r}")
        if not isinstance(self.sub_dim, int) or self.sub_dim < 1:
            raise ValueError(f"sub_dim must be a positive integer, got {self.sub_dim!r}")
        if self.head_dim % self.sub_dim:
            raise ValueError(f"head_dim {self.head_dim} is not a multiple of sub_dim "
                             f"{self.sub_dim}")
        if not isinstance(self.codebook_bits, int) or not 1 <= self.codebook_bits <= 24:
            raise ValueError(f"codebook_bits must be in [1, 24], got {self.codebook_bits!r}")
        for name in ("beta", "retrieval_fraction"):
            v = float(getattr(self, name))
            if not (0.0 <= v <= 1.0):  # also rejects NaN
                raise ValueError(f"{name} must lie in [0, 1], got {v!r}")
        if not isinstance(self.window, int):
            raise ValueError(f"window must be an integer, got {self.window!r}")
        if not isinstance(self.b, int) or abs(self.b) >= 1 << 24:
            raise ValueError(f"b must be an integer of magnitude below 2^24, got {self.b!r}")
        if not (float(self.rope_base) > 0.0 and math.isfinite(float(self.rope_base))):
            raise ValueError(f"rope_base must be positive and finite, got {self.rope_base!r}")
        if self.query_h is not None:
            shape = tuple(self.query_h.shape)
            if shape[-2:] != (self.sub_dim, self.sub_dim) or len(shape) not in (2, 3):
                raise ValueError(f"query_h must be {self.sub_dim} x {self.sub_dim} (per head), "
                                 f"got shape {shape}")
        if self.codebook is not None:
            shape = tuple(self.codebook.shape)
            if shape[-2:] != (self.n_centroids, self.sub_dim) or len(shape) not in (2, 3):
                raise ValueError(f"codebook must be {self.n_centroids} x {self.sub_dim} "
                                 f"(per head), got shape {shape}")
        return self

    def subvector_step(self, B: int, H: int, N: int, dtype, **kw):
        """The sub-vector step for B sequences of H heads and N cached
        tokens: retrieval fraction 0 when use_query_aware is off (every
        token then takes plain VQ)."""
        from .pipeline import A2ATSSubvectorStep

        self.validate()
        frac = self.retrieval_fraction if self.use_query_aware else 0.0
        return A2ATSSubvectorStep(B, H, N, self.head_dim, self.sub_dim, self.n_centroids,
                                  dtype, window=self.window, fraction=frac,
                                  rope_base=self.rope_base, beta=self.beta, **kw)

    def factor(self, H: int, device="cuda"):
        """L with query_h = L L^T for each of the H heads (a2ats_cholesky_factor
        on the device; a shared [sub_dim, sub_dim] query_h serves every head),
        or None without query_h.  Raises ValueError when query_h is not
        positive definite."""
        import torch

        from . import a2ats_cholesky_factor

        self.validate()
        if self.query_h is None:
            return None
        h = torch.as_tensor(self.query_h, dtype=torch.float32).to(device)
        if h.dim() == 2:
            h = h.expand(H, self.sub_dim, self.sub_dim)
        h = h.contiguous()
        if h.shape[0] != H:
            raise ValueError(f"query_h holds {h.shape[0]} heads, not {H}")
        L, info = a2ats_cholesky_factor(h)
        bad = info.cpu()
        if bool((bad != 0).any()):
            raise ValueError(f"query_h is not positive definite (failing minor per head: "
                             f"{bad.tolist()})")
        return L

    def byte_accounting(self, tokens: int) -> dict:
        """The page's byte accounting of `tokens` keys and values under
        these settings (a2ats_byte_accounting, host arithmetic)."""
        from . import a2ats_byte_accounting

        self.validate()
        return a2ats_byte_accounting(tokens, self.head_dim, self.sub_dim, self.codebook_bits)
