"""Shared helpers of the parity tests: tolerance checks and the top-k rule."""
from __future__ import annotations

import numpy as np
import torch

# tolerances on attention outputs (max-abs), per the parity bar of the build
TOL_F32 = 1e-4
TOL_BF16 = 2e-2
# Outputs are also held to a bound relative to the reference's largest magnitude: with
# the method's input recipe (cache rows N(0,1)/sqrt(c)) attention outputs are ~1e-3, so
# the absolute bound alone would pass an all-zero or mis-accumulated output.
REL_OUT = 1e-2
TOPK_GAP = 1e-3  # relative oracle score gap below which several top-k sets count as correct


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16 or t.dtype == torch.float8_e4m3fn:
        t = t.to(torch.float64)
    return t.numpy()


def max_abs(a, b) -> float:
    """Largest |a - b|; equal infinities count as equal, and a NaN on either side
    where the other side has none (or any NaN difference) counts as infinite."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        raise AssertionError(f"shape {a.shape} vs {b.shape}")
    if a.size == 0:
        return 0.0
    nan_a, nan_b = np.isnan(a), np.isnan(b)
    if np.any(nan_a != nan_b):
        return float("inf")
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.abs(np.where(both_inf | (nan_a & nan_b), 0.0, a - b))
    return float(np.max(d))


def out_close(got, ref, tol: float = TOL_BF16, rel: float = REL_OUT) -> bool:
    """An attention output is close to the reference when its max-abs error is within
    `tol` AND within `rel` of the reference's largest magnitude (a reference that is
    zero everywhere must be matched exactly)."""
    err = max_abs(got, ref)
    scale = float(np.max(np.abs(np.nan_to_num(np.asarray(ref, dtype=np.float64))))) if np.size(ref) else 0.0
    return err <= tol and err <= rel * scale


def assert_out_close(got, ref, tol: float = TOL_BF16, rel: float = REL_OUT, what: str = "output"):
    err = max_abs(got, ref)
    scale = float(np.max(np.abs(np.nan_to_num(np.asarray(ref, dtype=np.float64))))) if np.size(ref) else 0.0
    assert err <= tol, f"{what}: max-abs error {err:.3e} > {tol:.1e}"
    assert err <= rel * scale, f"{what}: max-abs error {err:.3e} > {rel:.0e} x max|ref| = {rel * scale:.3e}"


def check_topk_row(gpu_idx: np.ndarray, ref_scores: np.ndarray, visible: int, k: int, gap: float = TOPK_GAP):
    """Top-k parity for one query row.

    gpu_idx: the GPU's k indices (ascending, -1 padded).  ref_scores: the
    oracle's float64 scores of the visible entries.  The selected set must equal
    the oracle's where the oracle's k-th / (k+1)-th gap exceeds `gap` relative;
    otherwise the selected minimum must be >= the excluded maximum - gap*|max|.
    Returns "exact" or "relaxed" for reporting; raises AssertionError on failure.
    """
    take = min(k, visible)
    sel = gpu_idx[:take]
    assert (gpu_idx[take:] == -1).all(), "padding must be -1"
    if take == 0:
        return "exact"
    assert np.all(np.diff(sel) > 0), "indices must be strictly ascending"
    assert sel.min() >= 0 and sel.max() < visible, "index outside the visible entries"
    if take == visible:
        assert np.array_equal(sel, np.arange(visible))
        return "exact"
    s = ref_scores[:visible]
    order = np.lexsort((np.arange(visible), -s))  # score desc, index asc
    ref_set = np.sort(order[:take])
    kth, nxt = s[order[take - 1]], s[order[take]]
    scale = max(abs(kth), abs(nxt), 1e-30)
    if (kth - nxt) > gap * scale:
        assert np.array_equal(sel, ref_set), "top-k set differs from the oracle's with a clear score gap"
        return "exact"
    mask = np.zeros(visible, dtype=bool)
    mask[sel] = True
    excl_max = s[~mask].max()
    sel_min = s[mask].min()
    assert sel_min >= excl_max - gap * max(abs(excl_max), 1e-30), "selected set violates the relaxed top-k rule"
    return "relaxed"
