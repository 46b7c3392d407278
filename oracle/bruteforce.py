"""Membership of the allowed set by counting, with no sorting (small V only).

TEST INFRASTRUCTURE ONLY.  This is the predicate form of the filters, written
independently of ``oracle.filters`` (which reads prefixes off a sort), so that the
two can be checked against each other:

  * top-k: i is kept iff fewer than k tokens are strictly larger
      -- [blog] rejection sampling ("check how many tokens lie above the pivot");
  * top-p: i is kept iff the mass strictly above p_i is below p * M (or nothing
    is above it)
      -- [blog] rejection sampling, steps 1-2 ("q >= top_p needs another round,
         otherwise accept"); [explainer] Top-p;
  * min-p: p_i >= p_base * max
      -- [blog] Min-P;
  * top_k_first: the top-p test runs against F_k, the mass of the top-k items
      -- [explainer] filter order.
Zeros are never kept; invalid rows keep nothing.
"""
from __future__ import annotations

import math

import numpy as np


def members(p, top_k=None, top_p=None, min_p=None, order="joint") -> np.ndarray:
    p = [float(np.float32(x)) for x in np.asarray(p, dtype=np.float32)]
    V = len(p)
    if any(math.isnan(x) or x < 0 for x in p) or sum(p) <= 0:
        return np.zeros(0, np.int64)
    if top_p is not None and math.isnan(float(top_p)):
        return np.zeros(0, np.int64)
    if min_p is not None and math.isnan(float(min_p)):
        return np.zeros(0, np.int64)
    M = math.fsum(p)
    big = max(p)
    k_on = top_k is not None and 0 < int(top_k) < V
    p_on = top_p is not None and float(np.float32(top_p)) < 1.0
    m_on = min_p is not None and float(np.float32(min_p)) > 0.0

    def n_above(i):
        return sum(1 for x in p if x > p[i])

    def mass_above(i):
        return math.fsum(x for x in p if x > p[i])

    in_k = [p[i] > 0 and (not k_on or n_above(i) < int(top_k)) for i in range(V)]
    if order == "top_k_first" and k_on:
        ref_mass = math.fsum(p[i] for i in range(V) if in_k[i])
    else:
        ref_mass = M
    pp = float(np.float32(top_p)) if p_on else None
    kept = []
    for i in range(V):
        if p[i] <= 0 or not in_k[i]:
            continue
        if p_on and not (n_above(i) == 0 or mass_above(i) < pp * ref_mass):
            continue
        if m_on and not (p[i] >= float(np.float32(min_p)) * big):
            continue
        kept.append(i)
    return np.array(kept, np.int64)
