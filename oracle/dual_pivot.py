"""The dual-pivot rejection sampler, step by step as the pages state it.

TEST INFRASTRUCTURE ONLY.

Algorithm ([blog] "dual-pivot rejection sampling"; [explainer] "how dual pivot
shrinks the range"):
  f(x) = 1 iff threshold x already satisfies the filters.
  low <- 0, high <- max_i p_i, so that f(low) = 0 and f(high) = 1.
  repeat:
    draw j by inverse transform sampling over the tokens with p_i > low;
    pivot1 <- p_j, pivot2 <- (pivot1 + high) / 2;
    f(pivot1) = 1                -> return j;
    f(pivot1) = 0, f(pivot2) = 1 -> low <- pivot1, high <- pivot2;
    f(pivot1) = 0, f(pivot2) = 0 -> low <- pivot2.

The acceptance test at a threshold tau, written from the rejection-sampling
section of [blog] (count / remaining mass above the pivot) and the filter
definitions of [explainer]:
  f(tau) = [top-k: #{p > tau} < k]
         and [top-p: #{p > tau} = 0  or  sum_{p > tau} p < top_p * M']
         and [min-p: tau >= p_base * max]
with M' the row mass M (joint) or F_k, the mass of the k largest (top_k_first;
the draws then start from low = the largest value outside the top k, so only the
top-k items are ever drawn).

Inverse transform ([blog] "inverse transform sampling"; [explainer] "without
filters"): u ~ U[0,1), target = u * S(low) with S(low) = sum_{p > low} p, and the
token is the first j (index order) whose running sum over eligible tokens
exceeds the target.

Readings: the midpoint is rounded to float32 like the probabilities it is
compared with ("fp32"); "exact" keeps it rational for the Markov evaluation.
"single" is the one-pivot sampler of the [blog] rejection-sampling section (after a
rejection, low <- pivot1; no second pivot), kept for the ablation.
"Repeat steps 3 and 4" (garbled in [blog]) is read as "repeat from the draw".
A row is invalid when f(high) = 0 at the start (S empty) or when r_max draws pass
without acceptance.

``exact_output_law`` evaluates recurrence (star) of the [blog] proof exactly, with
rational arithmetic, over every path of the algorithm; the theorem says the result
is p_j / Z on S.
"""
from __future__ import annotations

from fractions import Fraction
from functools import lru_cache
from typing import Callable, Optional

import numpy as np

from . import filters
from .philox import sampler_uniform


class _Row:
    """Predicate data for one row, in float64 (``exact=False``) or rationals."""

    def __init__(self, p, top_k=None, top_p=None, min_p=None, order="joint", exact=False):
        p32 = np.asarray(p, dtype=np.float32)
        self.V = p32.size
        self.exact = exact
        conv = (lambda x: Fraction(float(x))) if exact else float
        self.p64 = p32.astype(np.float64)
        self.valid = filters.row_is_valid(p32)
        self.p = [conv(x) for x in p32] if self.valid else []
        self.order = order
        V = self.V
        self.k_on = top_k is not None and 0 < int(top_k) < V
        self.k = int(top_k) if self.k_on else None
        self.p_on = top_p is not None and float(np.float32(top_p)) < 1.0
        self.top_p = conv(np.float32(top_p)) if self.p_on else None
        self.m_on = min_p is not None and float(np.float32(min_p)) > 0.0
        if top_p is not None and np.isnan(float(top_p)):
            self.valid = False
        if min_p is not None and np.isnan(float(min_p)):
            self.valid = False
        if not self.valid:
            return
        self.high0 = max(self.p)
        self.M = sum(self.p, conv(0))
        self.t_min = conv(np.float32(min_p)) * self.high0 if self.m_on else None
        self.low0 = conv(0)
        self.Mp = self.M
        if order == "top_k_first" and self.k_on:
            desc = sorted(self.p, reverse=True)
            head = [x for x in desc[: self.k] if x > 0]
            self.Mp = sum(head, conv(0))
            rest = [x for x in desc[self.k:] if x > 0]
            self.low0 = rest[0] if rest else conv(0)

    def count_mass_above(self, tau):
        if self.exact:
            above = [x for x in self.p if x > tau]
            return len(above), sum(above, Fraction(0))
        mask = self.p64 > float(tau)
        return int(mask.sum()), float(self.p64[mask].sum())

    def f(self, tau) -> bool:
        cnt, mass = self.count_mass_above(tau)
        if self.k_on and not cnt < self.k:
            return False
        if self.p_on and not (cnt == 0 or mass < self.top_p * self.Mp):
            return False
        if self.m_on and not tau >= self.t_min:
            return False
        return True

    def midpoint(self, a, b, mode: str):
        if mode == "exact":
            return (a + b) / 2
        s = np.float32(np.float32(float(a)) + np.float32(float(b))) * np.float32(0.5)
        return Fraction(float(s)) if self.exact else float(s)


def three_cases(row: _Row, pivot1, high, midpoint: str):
    """The case analysis after a draw with value pivot1.

    Returns None when the draw is accepted (case 1), else the next (low, high):
    (pivot1, pivot2) when f(pivot2) = 1 (case 2), (pivot2, high) otherwise (case 3).
    """
    if row.f(pivot1):
        return None
    if midpoint == "single":
        return pivot1, high
    pivot2 = row.midpoint(pivot1, high, midpoint)
    if row.f(pivot2):
        return pivot1, pivot2
    return pivot2, high


def draw_inverse_transform(p64: np.ndarray, low: float, u: float) -> int:
    """First index whose running sum over {p > low} exceeds u * S(low).

    If rounding leaves no such index, the last eligible index is taken (the
    monotonicity guard of [blog] "implementation details").
    """
    masked = np.where(p64 > low, p64, 0.0)
    cum = np.cumsum(masked)
    target = u * cum[-1]
    hit = np.nonzero((cum > target) & (masked > 0))[0]
    if hit.size:
        return int(hit[0])
    return int(np.nonzero(masked > 0)[0][-1])


def sample(p, top_k=None, top_p=None, min_p=None, order="joint",
           uniform: Optional[Callable[[int], float]] = None, r_max: int = 256,
           midpoint: str = "fp32"):
    """Run the sampler on one row.  Returns (token, valid, rounds).

    ``uniform(r)`` is the uniform of round r (0-based); ``rounds`` counts draws.
    """
    row = _Row(p, top_k, top_p, min_p, order, exact=False)
    if not row.valid:
        return -1, False, 0
    low, high = row.low0, row.high0
    if not row.f(high):
        return -1, False, 0
    for r in range(r_max):
        j = draw_inverse_transform(row.p64, low, uniform(r))
        nxt = three_cases(row, row.p[j], high, midpoint)
        if nxt is None:
            return j, True, r + 1
        low, high = nxt
    return -1, False, r_max


def sample_philox(p, top_k=None, top_p=None, min_p=None, order="joint", *,
                  seed: int, offset: int, row: int, r_max: int = 256, midpoint: str = "fp32"):
    """``sample`` driven by the Philox stream of output row ``row`` (see oracle.philox)."""
    return sample(p, top_k, top_p, min_p, order,
                  uniform=lambda r: sampler_uniform(seed, offset, row, r), r_max=r_max, midpoint=midpoint)


def exact_output_law(p, top_k=None, top_p=None, min_p=None, order="joint",
                     midpoint: str = "exact") -> dict:
    """Pr[output = j] for every j, by exact evaluation of recurrence (star).

    From a state (low, high) the next draw picks i with probability
    p_i / S(low) among p_i > low; acceptance ends the path, otherwise the state
    moves as the three cases say.  Every failure raises ``low`` past a token, so
    the recursion is finite.  Returns {} for an invalid row.
    """
    row = _Row(p, top_k, top_p, min_p, order, exact=True)
    if not row.valid or not row.f(row.high0):
        return {}

    @lru_cache(maxsize=None)
    def law(low: Fraction, high: Fraction):
        elig = [i for i in range(row.V) if row.p[i] > low]
        S = sum((row.p[i] for i in elig), Fraction(0))
        out: dict = {}
        for i in elig:
            w = row.p[i] / S
            nxt = three_cases(row, row.p[i], high, midpoint)
            if nxt is None:
                out[i] = out.get(i, Fraction(0)) + w
                continue
            sub = law(*nxt)
            for j, q in sub.items():
                out[j] = out.get(j, Fraction(0)) + w * q
        return out

    return dict(law(row.low0, row.high0))


def max_draws(p, top_k=None, top_p=None, min_p=None, order="joint", midpoint: str = "fp32") -> int:
    """The largest number of draws any run of the sampler can take on this row.

    The same walk over the algorithm's states (low, high) as ``exact_output_law``:
    from a state every eligible token (p_i > low) is drawn with positive
    probability; an accepted draw ends the path after one draw, a rejected one
    continues from the state the three cases give.  Returns the longest path, 0 for
    an invalid row or an empty S.  Exact rationals, so the answer does not depend on
    summation order; ``midpoint`` as in ``sample`` ("fp32" is the kernels' rule).
    """
    row = _Row(p, top_k, top_p, min_p, order, exact=True)
    if not row.valid or not row.f(row.high0):
        return 0

    @lru_cache(maxsize=None)
    def longest(low: Fraction, high: Fraction) -> int:
        best = 0
        for i in range(row.V):
            if not row.p[i] > low:
                continue
            nxt = three_cases(row, row.p[i], high, midpoint)
            best = max(best, 1 if nxt is None else 1 + longest(*nxt))
        return best

    return longest(row.low0, row.high0)
