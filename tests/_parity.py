"""Helpers for the GPU parity tests: exact decoding, tolerance checks and the
near-tie exemption rule (codes and retrieval sets must match the oracle
bit for bit except on rows whose oracle top-2 gap is below 1e-5)."""
import numpy as np
import torch

TIE = 1e-5


def f64(t) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def dev(t, device="cuda"):
    return t.to(device).contiguous()


def ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Spacing of the storage format at |x| (normal range)."""
    mant = {torch.bfloat16: 7, torch.float16: 10, torch.float32: 23}[dtype]
    tiny = {torch.bfloat16: 2.0 ** -126, torch.float16: 2.0 ** -14, torch.float32: 2.0 ** -126}[dtype]
    a = np.maximum(np.abs(x), tiny)
    return 2.0 ** (np.floor(np.log2(a)) - mant)


def rne(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).to(torch.float64).numpy()


def assert_rows_close(got, want, rel=1e-3):
    """max |got - want| over a row <= rel * max |want| of that row."""
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    scale = np.abs(want).max(axis=-1, keepdims=True)
    err = np.abs(got - want).max(axis=-1, keepdims=True)
    bad = err > rel * np.maximum(scale, 1e-30)
    assert not bad.any(), f"{bad.sum()} rows off; worst {float((err / np.maximum(scale, 1e-30)).max()):.3g}"
    return float((err / np.maximum(scale, 1e-30)).max())


def assert_storage_close(got, want, dtype, rot_err=2e-6):
    """A rotated key stored in a 16-bit format is at most one unit in the last
    place from the oracle's fp64 value rounded to nearest even, plus the fp32
    rotation's own error, rot_err times the row's largest element (it decides
    only where the two terms of a rotated element cancel to far below the
    row's scale); fp32 storage within 1e-5 of the row's largest element."""
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    if dtype == torch.float32:
        return assert_rows_close(got, want, rel=1e-5)
    r = rne(want, dtype)
    slack = rot_err * np.abs(want).max(axis=-1, keepdims=True)
    bad = np.abs(got - r) > ulp(r, dtype) + slack + 1e-30
    assert not bad.any(), f"{bad.sum()} elements more than 1 ulp from the rounded oracle"
    return 0.0


def check_codes(gpu, want, gap, what="codes"):
    """Codes equal the oracle's on every row whose relative top-2 gap is at
    least TIE; returns (mismatches on exempt rows, exempt rows).  A NaN gap
    (one centroid: the second distance is infinite) exempts nothing."""
    gpu, want, gap = np.asarray(gpu), np.asarray(want), np.asarray(gap)
    bad = (gpu != want) & ~(gap < TIE)
    assert not bad.any(), (f"{what}: {bad.sum()} of {len(want)} non-exempt rows differ, "
                           f"first at {np.flatnonzero(bad)[:5]} (gap {gap[bad][:5]})")
    return int(((gpu != want) & (gap < TIE)).sum()), int((gap < TIE).sum())


def check_split(perm, count, n, k_want, scores, kth):
    """Retrieval set of one (b, h): exact size, disjoint and covering, both
    halves ascending, and membership equal to the oracle's except for rows
    whose score is within TIE of the n_r-th largest."""
    perm = np.asarray(perm)[:n]
    assert count == k_want
    assert sorted(perm.tolist()) == list(range(n))
    ret, bulk = perm[:count], perm[count:]
    assert (np.diff(ret) > 0).all() and (np.diff(bulk) > 0).all()
    s = np.asarray(scores)
    if count:
        must_in = np.flatnonzero(s > kth + TIE)
        must_out = np.flatnonzero(s < kth - TIE)
        inset = np.zeros(n, bool)
        inset[ret] = True
        assert inset[must_in].all(), "a clearly-above-threshold row is missing"
        assert not inset[must_out].any(), "a clearly-below-threshold row was retrieved"
