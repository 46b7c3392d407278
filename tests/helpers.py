"""Shared test utilities: oracle-side expectations and statistics.

Only tests import this module.  Expected values come from ``oracle/``; the CUDA
results come from the library under test.
"""
from __future__ import annotations

import math
import os
import subprocess
import sys

import numpy as np

from oracle import filters

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GUARD = 1e-5        # distance of decisive top-p prefix masses from the target
GUARD_DEEP = 2e-6   # used where the boundary token itself is lighter than 2 * GUARD


def ensure_built() -> str:
    lib = os.path.join(ROOT, "min_sampling_gb300", "libfs_sampling.so")
    if not os.path.exists(lib):
        subprocess.run([sys.executable, "-m", "min_sampling_gb300.build"], cwd=ROOT, check=True)
    return lib


def guard_accept(param_sets, delta: float = GUARD):
    """Accept callback for workloads: every (k, p, minp, order) use of row i must keep
    its top-p boundary at least `delta` away from the target.  A use may carry its own
    delta as a fifth element."""
    def accept(i, row):
        for ps in param_sets(i):
            d = ps[4] if len(ps) > 4 else delta
            if filters.topp_boundary_margin(row, *ps[:4]) < d:
                return False
        return True
    return accept


def allowed_masks(probs, top_k, top_p, min_p, order, indices=None):
    """Boolean [B_out, V] allowed-set masks and [B_out] validity from the oracle.
    Output rows that share an input row and parameters reuse one computation."""
    b_out = len(top_k) if top_k is not None else (len(indices) if indices is not None else probs.shape[0])
    V = probs.shape[1]
    masks = np.zeros((b_out, V), bool)
    valid = np.zeros(b_out, bool)
    cache = {}
    for b in range(b_out):
        r = int(indices[b]) if indices is not None else b
        k = None if top_k is None else int(top_k[b])
        p = None if top_p is None else float(top_p[b])
        m = None if min_p is None else float(min_p[b])
        key = (r, k, p, m)
        if key not in cache:
            if 0 <= r < probs.shape[0]:
                cache[key] = filters.allowed_set(probs[r], k, p, m, order)
            else:
                cache[key] = np.zeros(0, np.int64)
        S = cache[key]
        masks[b, S] = True
        valid[b] = S.size > 0
    return masks, valid


def tv_distance(counts: np.ndarray, pt: np.ndarray) -> float:
    n = counts.sum()
    return 0.5 * float(np.abs(counts / n - pt).sum())


def expected_null_tv(pt: np.ndarray, n: int) -> float:
    """E[TV] of an exact sampler of pt with n draws (normal approximation)."""
    pt = pt[pt > 0]
    return 0.5 * float(np.sum(np.sqrt(2.0 * pt * (1.0 - pt) / (math.pi * n))))


def draws_for_tv(pt: np.ndarray, target: float = 0.002, lo: int = 10 ** 6, hi: int = 1 << 24) -> int:
    """Smallest n (>= lo, <= hi) whose null E[TV] is at most `target`."""
    pt = pt[pt > 0]
    s = 0.5 * float(np.sum(np.sqrt(2.0 * pt * (1.0 - pt) / math.pi)))
    n = int(math.ceil((s / target) ** 2))
    return int(min(max(n, lo), hi))


def chi2_pvalue(counts: np.ndarray, pt: np.ndarray) -> float:
    """Pearson chi-square p-value; cells with expected count < 5 are pooled."""
    from scipy.stats import chi2

    n = counts.sum()
    exp = pt * n
    keep = exp >= 5
    obs_k, exp_k = counts[keep].astype(np.float64), exp[keep]
    rest_o, rest_e = counts[~keep].sum(), exp[~keep].sum()
    if rest_e >= 5:
        obs_k = np.append(obs_k, rest_o)
        exp_k = np.append(exp_k, rest_e)
    elif rest_o > 0 and obs_k.size:
        obs_k[-1] += rest_o
        exp_k[-1] += rest_e
    dof = obs_k.size - 1
    if dof <= 0:
        return 1.0
    stat = float(np.sum((obs_k - exp_k) ** 2 / exp_k))
    return float(chi2.sf(stat, dof))
