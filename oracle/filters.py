"""Allowed sets and renormalised outputs, written out from their definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every computation is in
float64 over the float32 inputs (each float32 converts to float64 exactly), using a
descending sort of the row as the plain way to read off prefixes.

Definitions followed:
  * p~_i = p_i / sum_{j in S} p_j on S, 0 elsewhere
      -- [explainer] "what the sampling pipeline computes".
  * S_k = the k largest; k = V means no filter
      -- [blog] Top-K; [explainer] Top-k.
  * S_p = the smallest descending prefix whose cumulative mass reaches p:
    m = min{r : F_r >= p * M}
      -- [explainer] Top-p (the ">=" form); [blog] Top-P.
  * S_min = {i : p_i >= p_base * max_j p_j}
      -- [blog] Min-P; [explainer] Min-p.
  * joint = all filters checked together; top_k_first = top-k, then top-p inside
    the k items with their cumulative mass renormalised
      -- [explainer] "the order of top-k and top-p changes the distribution";
         [blog] footnote 1.
  * renorm: keep x >= t where t is the largest threshold with count(x >= t) >= k
    (top-k) or mass(x >= t) >= p (top-p), then divide by the kept mass
      -- [drill] sections 2-4.

Readings where the pages are silent or loose (each is listed in the design notes):
  * top-p is measured against the row's own total M (p * M), so unnormalised rows
    behave as their normalised version; top_p >= 1 keeps every positive entry,
    top_p <= 0 keeps the arg-max only (the sort path's "keep at least one").
  * top_k <= 0 or top_k >= V: no top-k filter.  min_p <= 0: no min-p filter;
    min_p > 1 empties S (row reported invalid).
  * zeros are never in S; a row with a NaN, a negative entry or zero total mass
    is invalid, as is a row whose S is empty.
  * top_k_first measures top-p against F_k, the mass of the k kept items.
  * joint is the intersection of the three filters, each on the original row.
  * min-p threshold: the product p_base * max of two float32 values, exact in
    float64.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

ORDERS = ("joint", "top_k_first")


def as64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def row_is_valid(p) -> bool:
    """No NaN, no negative entry and a positive total ([explainer] degenerate rows)."""
    p = as64(p)
    if np.isnan(p).any() or (p < 0).any():
        return False
    return bool(p.sum() > 0.0)


def descending_positive(p) -> np.ndarray:
    """Indices of the positive entries, largest value first (ties by lower index)."""
    p = as64(p)
    pos = np.nonzero(p > 0)[0]
    order = np.lexsort((pos, -p[pos]))
    return pos[order]


def _k_active(top_k, V: int) -> bool:
    return top_k is not None and 0 < int(top_k) < V


def _p_active(top_p) -> bool:
    return top_p is not None and float(top_p) < 1.0


def _minp_active(min_p) -> bool:
    return min_p is not None and float(min_p) > 0.0


def top_p_prefix_len(sorted_vals: np.ndarray, top_p: float, mass: float) -> int:
    """m = min{r : F_r >= top_p * mass} over descending values; 1 when top_p <= 0."""
    if float(top_p) <= 0.0:
        return min(1, sorted_vals.size)
    target = float(np.float32(top_p)) * mass
    F = np.cumsum(sorted_vals)
    hit = np.nonzero(F >= target)[0]
    return int(hit[0]) + 1 if hit.size else int(sorted_vals.size)


def min_p_threshold(p, min_p: float) -> float:
    """p_base * max_j p_j, exact in float64 for float32 operands."""
    return float(np.float32(min_p)) * float(as64(p).max())


def allowed_set(p, top_k=None, top_p=None, min_p=None, order: str = "joint") -> np.ndarray:
    """The allowed set S as a sorted array of token indices (empty if the row is invalid)."""
    if order not in ORDERS:
        raise ValueError(order)
    p64 = as64(p)
    V = p64.size
    if not row_is_valid(p64):
        return np.zeros(0, np.int64)
    if top_p is not None and math.isnan(float(top_p)):
        return np.zeros(0, np.int64)
    if min_p is not None and math.isnan(float(min_p)):
        return np.zeros(0, np.int64)
    desc = descending_positive(p64)
    vals = p64[desc]
    n = desc.size
    M = float(p64.sum())

    n_k = min(int(top_k), n) if _k_active(top_k, V) else n
    if _minp_active(min_p):
        t_min = min_p_threshold(p64, min_p)
        n_min = int(np.count_nonzero(vals >= t_min))
    else:
        n_min = n

    if order == "joint":
        n_p = top_p_prefix_len(vals, top_p, M) if _p_active(top_p) else n
        m = min(n_k, n_p, n_min)
    else:
        head = vals[:n_k]
        F_k = float(head.sum())
        n_p = top_p_prefix_len(head, top_p, F_k) if _p_active(top_p) else n_k
        m = min(n_k, n_p, n_min)
    return np.sort(desc[:m])


def filtered_distribution(p, top_k=None, top_p=None, min_p=None, order="joint"):
    """(p~ as a float64 vector of length V, valid flag)."""
    p64 = as64(p)
    S = allowed_set(p64, top_k, top_p, min_p, order)
    out = np.zeros(p64.size, np.float64)
    if S.size == 0:
        return out, False
    Z = float(p64[S].sum())
    if not Z > 0:
        return out, False
    out[S] = p64[S] / Z
    return out, True


def cut_value(p, top_k=None, top_p=None, min_p=None, order="joint") -> float:
    """tau*: the smallest threshold tau at which the acceptance test f(tau) holds.

    Each filter switches on at its own cut: top-k at the k-th largest value,
    top-p at the m-th largest (the last member of the nucleus), min-p at
    p_base * max.  The test is their conjunction, so tau* is the largest active
    cut.  Used only for the round-count bound.
    """
    p64 = as64(p)
    V = p64.size
    vals = p64[descending_positive(p64)]
    cuts = [0.0]
    if order == "top_k_first" and _k_active(top_k, V):
        vals = vals[: min(int(top_k), vals.size)]
        Mp = float(vals.sum())
    else:
        Mp = float(p64.sum())
    if _k_active(top_k, V) and int(top_k) <= vals.size:
        cuts.append(float(vals[int(top_k) - 1]))
    if _p_active(top_p):
        cuts.append(float(vals[top_p_prefix_len(vals, top_p, Mp) - 1]))
    if _minp_active(min_p):
        cuts.append(min_p_threshold(p64, min_p))
    return max(cuts)


def round_bound_terms(p, top_k=None, top_p=None, min_p=None, order="joint"):
    """The two limits on the number of draws of the dual-pivot sampler for one row.

    Facts from [blog] dual-pivot section / [explainer] "how dual pivot shrinks the
    range":
      * every failed round raises `low` past the drawn (rejected) token, so the
        failures are at most the number of rejectable tokens above the starting
        `low` (``by_count`` = that number + 1 draws);
      * every failed round at least halves high - low, and the round that ends
        the search needs high - low below tau* - a (a = the largest rejectable
        value, tau* = the cut of the acceptance test, ``cut_value``), so the
        failures are at most log2(high0 / (tau* - a)) rounded up, plus 2 for the
        float32 rounding of the midpoint (``by_halving`` = 3 + that log).
    Returns (by_count, by_halving), or None when S is empty; (1, 1) when no token
    can be rejected.
    """
    p64 = as64(p)
    S = allowed_set(p64, top_k, top_p, min_p, order)
    if S.size == 0:
        return None
    V = p64.size
    desc = descending_positive(p64)
    if order == "top_k_first" and _k_active(top_k, V):
        pool = desc[: min(int(top_k), desc.size)]
    else:
        pool = desc
    inS = np.zeros(V, bool)
    inS[S] = True
    rejectable = pool[~inS[pool]]
    if rejectable.size == 0:
        return 1, 1
    a = float(p64[rejectable].max())
    tau = cut_value(p64, top_k, top_p, min_p, order)
    hi0 = float(p64.max())
    by_count = rejectable.size + 1
    gap = tau - a
    by_halving = 3 + int(math.ceil(math.log2(hi0 / gap))) if gap > 0 else by_count
    return int(by_count), int(by_halving)


def round_bound(p, top_k=None, top_p=None, min_p=None, order="joint") -> int:
    """Upper bound on the number of draws of the dual-pivot sampler for one row:
    the smaller of the two limits of ``round_bound_terms`` (0 when S is empty)."""
    t = round_bound_terms(p, top_k, top_p, min_p, order)
    return 0 if t is None else int(min(t))


def topp_boundary_margin(p, top_k=None, top_p=None, min_p=None, order="joint") -> float:
    """Distance of the decisive top-p prefix masses from the top-p target.

    The top-p test compares F_r (the mass of the r largest) with p * M'.  Only the
    prefixes r = m-1 and r = m around the crossing can be misjudged by rounding,
    and only while the other filters still pass at that rank.  Returns
    min |F_r - p M'| over those r, or +inf when top-p never decides.  Inputs whose
    margin is below the agreed guard (1e-5) are redrawn by the tests.
    """
    p64 = as64(p)
    V = p64.size
    if not row_is_valid(p64) or not _p_active(top_p) or float(top_p) <= 0.0:
        return math.inf
    desc = descending_positive(p64)
    vals = p64[desc]
    n = vals.size
    if order == "top_k_first" and _k_active(top_k, V):
        vals = vals[: min(int(top_k), n)]
        Mp = float(vals.sum())
        other = vals.size
    else:
        Mp = float(p64.sum())
        other = min(int(top_k), n) if _k_active(top_k, V) else n
    if _minp_active(min_p):
        other = min(other, int(np.count_nonzero(vals >= min_p_threshold(p64, min_p))))
    target = float(np.float32(top_p)) * Mp
    F = np.concatenate(([0.0], np.cumsum(vals)))  # F[r] = mass of the r largest
    m = top_p_prefix_len(vals, top_p, Mp)
    margin = math.inf
    for r in (m - 1, m):
        if 0 <= r <= other and r < F.size:
            margin = min(margin, abs(F[r] - target))
    return margin


# ---------------------------------------------------------------------------
# Filter-only outputs ([drill] sections 2-4, [explainer] "filter / renormalise only").
# ---------------------------------------------------------------------------

def top_k_threshold(p, k: int) -> float:
    """Largest t with count(x >= t) >= k (0 when no filter applies)."""
    p64 = as64(p)
    V = p64.size
    if not (0 < int(k) < V):
        return 0.0
    vals = np.sort(p64)[::-1]
    return float(vals[int(k) - 1])


def top_k_renorm(p, k: int):
    """(renormalised float64 row, valid) for top_k_renorm_probs."""
    p64 = as64(p)
    out = np.zeros_like(p64)
    if not row_is_valid(p64):
        return out, False
    t = top_k_threshold(p64, k)
    keep = p64 >= t
    out[keep] = p64[keep] / p64[keep].sum()
    return out, True


def top_p_threshold(p, top_p: float) -> float:
    """Largest t with mass(x >= t) >= top_p * M; 0 when top_p >= 1; max when top_p <= 0."""
    p64 = as64(p)
    if float(top_p) >= 1.0:
        return 0.0
    vals = np.sort(p64[p64 > 0])[::-1]
    m = top_p_prefix_len(vals, top_p, float(p64.sum()))
    return float(vals[m - 1])


def top_p_renorm(p, top_p: float):
    """(renormalised float64 row, valid) for top_p_renorm_probs."""
    p64 = as64(p)
    out = np.zeros_like(p64)
    if not row_is_valid(p64) or math.isnan(float(top_p)):
        return out, False
    t = top_p_threshold(p64, top_p)
    keep = p64 >= t
    out[keep] = p64[keep] / p64[keep].sum()
    return out, True


def top_k_mask_logits(z, k: int):
    """(masked float32 logits, valid): the k largest kept, the rest -inf.

    A row holding a NaN is invalid and comes back all -inf.
    """
    z = np.asarray(z, dtype=np.float32)
    V = z.size
    if np.isnan(z).any():
        return np.full(V, -np.inf, np.float32), False
    if not (0 < int(k) < V):
        return z.copy(), True
    t = np.sort(z.astype(np.float64))[::-1][int(k) - 1]
    return np.where(z.astype(np.float64) >= t, z, np.float32(-np.inf)).astype(np.float32), True


def softmax(z, temperature: float = 1.0) -> np.ndarray:
    """p = softmax(z / T) in float64 ([explainer] the sampling pipeline: temperature
    then softmax before the filters), from the float32 logits converted exactly:
    exp((z_i - max z) / T) / sum_j exp((z_j - max z) / T).  -inf logits get 0."""
    z64 = np.asarray(z, dtype=np.float32).astype(np.float64)
    e = np.exp((z64 - z64.max()) / float(temperature))
    return e / e.sum()
