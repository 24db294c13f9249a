"""Oracle for the host-side scheduling half of the AdaptiveLoad technical summary, section
2.A: the dual-constraint bucket size with a real exponent, the Shape-Benchmarking fit of
the step-time model t = a + b * B * S^p, and the compute-load coefficient of variation a
bucketing rule leaves (the load-balance figure of the summary's results).

Test infrastructure only (plain Python / numpy, slow, written to be checked by eye); the
library's implementation lives in the package and shares nothing with this file.
"""
from __future__ import annotations

import math
from decimal import Decimal, getcontext
from typing import List, Sequence, Tuple

import numpy as np

from .bucket import bucket_batch


def bucket_batch_real(S: int, M_mem: int, M_comp: int, p: float) -> Tuple[int, bool]:
    """B = max(1, min(floor(M_mem / S), floor(M_comp / S^p))) with S^p evaluated in 60-digit
    decimal arithmetic from the exact binary value of p. Returns (B, near) where `near` says
    M_comp / S^p lies within 1e-12 (relative) of an integer, where a double-precision
    evaluation may land on either side."""
    if p == int(p) and 1 <= p <= 64:
        return bucket_batch(S, M_mem, M_comp, int(p)), False
    getcontext().prec = 60
    sp = (Decimal(p) * Decimal(S).ln()).exp()
    q = Decimal(M_comp) / sp
    k = int(q.to_integral_value(rounding="ROUND_FLOOR"))
    frac_dist = min(q - k, k + 1 - q)
    near = frac_dist <= q * Decimal("1e-12")
    return max(1, min(M_mem // S, k)), bool(near)


def _linear_fit(u: np.ndarray, t: np.ndarray) -> Tuple[float, float, float]:
    """Least squares t ~ a + b u by numpy's lstsq; returns a, b and the residual sum of squares."""
    A = np.stack([np.ones_like(u), u], axis=1)
    (a, b), *_ = np.linalg.lstsq(A, t, rcond=None)
    r = t - a - b * u
    return float(a), float(b), float(np.dot(r, r))


def fit_step_cost(B: Sequence[int], S: Sequence[int], t: Sequence[float], p_lo: float, p_hi: float,
                  t_budget: float) -> dict:
    """Fit t = a + b * B * S^p: for each p on a grid the model is linear in (a, b); take the p
    of least residual, then search grids 100x finer around it, three times."""
    B = np.asarray(B, dtype=np.float64)
    S = np.asarray(S, dtype=np.float64)
    t = np.asarray(t, dtype=np.float64)

    def rss(p):
        return _linear_fit(B * S ** p, t)[2]

    lo, hi = p_lo, p_hi
    best = lo
    for _ in range(4):
        grid = np.linspace(lo, hi, 2001)
        vals = [rss(p) for p in grid]
        j = int(np.argmin(vals))
        best = float(grid[j])
        step = (hi - lo) / 2000
        lo, hi = max(p_lo, best - step), min(p_hi, best + step)
    a, b, r = _linear_fit(B * S ** best, t)
    m_comp = math.floor((t_budget - a) / b) if (b > 0 and t_budget > a) else 0
    return {"a": a, "b": b, "p": best, "rms": math.sqrt(r / len(t)), "M_comp": float(m_comp)}


def batches_of(lengths: Sequence[int], buckets: Sequence[int], M_mem: int, M_comp: int, p: float,
               rule: int) -> List[Tuple[int, int]]:
    """The (bucket length, samples) of every batch: each sample goes to the smallest bucket
    that holds it; a bucket's samples, in order, fill batches of its size (rule 0: the
    equal-token size max(1, M_mem // S); rule 1: the dual constraint), the last partial."""
    per_bucket = {S: 0 for S in buckets}
    for L in lengths:
        S = min(b for b in buckets if b >= L)
        per_bucket[S] += 1
    out = []
    for S in buckets:
        c = per_bucket[S]
        size = max(1, M_mem // S) if rule == 0 else bucket_batch_real(S, M_mem, M_comp, p)[0]
        while c > 0:
            k = min(size, c)
            out.append((S, k))
            c -= k
    return out


def bucket_load_cv(lengths, buckets, M_mem, M_comp, p, rule) -> dict:
    """Population coefficient of variation of the batch costs k * S^p."""
    costs = [k * float(S) ** p for S, k in batches_of(lengths, buckets, M_mem, M_comp, p, rule)]
    mean = math.fsum(costs) / len(costs)
    var = math.fsum((c - mean) ** 2 for c in costs) / len(costs)
    return {"cv": math.sqrt(var) / mean, "batches": len(costs), "mean": mean}
