"""Sort-based reference sampler: the timed CPU baseline.

TEST INFRASTRUCTURE ONLY.  It follows the sort pipeline the pages describe as the
traditional path ([blog] the PyTorch top-k/top-p example; [explainer] "why the
sorting path is expensive"): sort the row, build the allowed set from prefixes,
renormalise, and draw once by inverse transform over the float64 cumulative sum,
with numpy's own PCG64 generator.  It is the oracle as it stands (``filters``
plus one draw), never tuned for speed.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from . import filters


def sample_row(p, top_k, top_p, min_p, order, rng: np.random.Generator):
    S = filters.allowed_set(p, top_k, top_p, min_p, order)
    if S.size == 0:
        return -1, False
    vals = filters.as64(p)[S]
    desc = np.argsort(-vals, kind="stable")
    cdf = np.cumsum(vals[desc])
    j = int(np.searchsorted(cdf, rng.random() * cdf[-1], side="right"))
    return int(S[desc[min(j, S.size - 1)]]), True


def sample_rows(probs, top_k, top_p, min_p, order="joint", indices: Optional[np.ndarray] = None,
                rng: Optional[np.random.Generator] = None):
    rng = rng if rng is not None else np.random.default_rng()
    b_out = len(top_k)
    tok = np.full(b_out, -1, np.int64)
    ok = np.zeros(b_out, bool)
    for b in range(b_out):
        r = int(indices[b]) if indices is not None else b
        k = None if top_k is None else int(top_k[b])
        pp = None if top_p is None else float(top_p[b])
        mp = None if min_p is None else float(min_p[b])
        tok[b], ok[b] = sample_row(probs[r], k, pp, mp, order, rng)
    return tok, ok
