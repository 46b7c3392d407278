"""Sampling from logits with the softmax fused into the kernel
(fs_top_k_top_p_sampling_from_logits) against the oracle's float64 softmax and
filters: the law on small rows, membership on full-size rows, invalid rows."""
import numpy as np
import pytest

import workloads
from oracle import filters
from tests.helpers import (allowed_masks, chi2_pvalue, draws_for_tv, ensure_built, expected_null_tv, guard_accept,
                           tv_distance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ms():
    ensure_built()
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import min_sampling_gb300
    return min_sampling_gb300


def _logit_rows(n, V, sigma, seed, uses, temperature=1.0):
    """Tie-free float32 logit rows whose softmax keeps every top-p boundary away from
    its target (the oracle's guard, on the float64 softmax)."""
    acc = guard_accept(uses)
    rows = []
    for i in range(n):
        for att in range(64):
            rng = workloads.row_rng(seed, i, att)
            z, _ = workloads.detie(rng.normal(0, sigma, V).astype(np.float32), positive_only=False)
            if acc(i, filters.softmax(z, temperature)):
                break
        rows.append(z)
    return np.stack(rows)


CASES = [(None, None, None, "joint", 1.0), (10, 0.9, None, "joint", 0.7), (50, 0.95, 0.1, "top_k_first", 1.5),
         (None, 0.5, None, "joint", 1.0), (1, None, None, "joint", 2.0)]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_law_on_small_rows(ms, case):
    import torch
    k, p, mp, order, T = CASES[case]
    Z = _logit_rows(2, 1024, 2.0, 700 + case, lambda i: [(k, p, mp, order)] if p is not None else [], T)
    Zt = torch.from_numpy(Z).cuda()
    for r in range(2):
        pt, ok = filters.filtered_distribution(filters.softmax(Z[r], T), k, p, mp, order)
        assert ok
        n = draws_for_tv(pt)
        idx = torch.from_numpy(np.full(n, r, np.int32)).cuda()
        tok, valid = ms.top_k_top_p_sampling_from_logits(
            Zt, T, k, p, mp, order, idx, seed=31 + case, offset=r)
        tok, valid = tok.cpu().numpy(), valid.cpu().numpy()
        assert valid.all() and (pt[tok] > 0).all(), "a draw outside S"
        counts = np.bincount(tok, minlength=1024).astype(np.float64)
        tv = tv_distance(counts, pt)
        assert tv <= 0.005, (case, r, tv, expected_null_tv(pt, n))
        assert chi2_pvalue(counts, pt) > 1e-3, (case, r)


def test_full_size_membership(ms):
    """B=64, V=151936 logits (z ~ N(0, 9)), top-k 50 + top-p 0.9 in both orders, T = 1."""
    import torch
    uses = lambda i: [(50, 0.9, None, "top_k_first"), (50, 0.9, None, "joint")]
    Z = _logit_rows(64, 151936, 3.0, 777, uses)
    P = np.stack([filters.softmax(z) for z in Z])
    Zt = torch.from_numpy(Z).cuda()
    k = np.full(64, 50, np.int32)
    p = np.full(64, 0.9, np.float32)
    for order in ("top_k_first", "joint"):
        masks, vref = allowed_masks(P, k, p, None, order)
        for call in range(3):
            tok, valid = ms.top_k_top_p_sampling_from_logits(Zt, None, torch.from_numpy(k).cuda(),
                                                             torch.from_numpy(p).cuda(), None, order,
                                                             seed=3, offset=call)
            tok, valid = tok.cpu().numpy(), valid.cpu().numpy()
            assert np.array_equal(valid.astype(bool), vref)
            assert masks[np.arange(64), tok].all(), "a draw outside S"


def test_invalid_rows_and_neg_inf(ms):
    import torch
    Z = _logit_rows(1, 300, 1.0, 5, lambda i: [])[0]
    rows = np.stack([Z, Z, Z, Z, Z])
    rows[1, 7] = np.nan
    rows[2, 9] = np.inf
    rows[4, ::2] = -np.inf   # the even tokens can never be drawn
    T = np.array([1.0, 1.0, 1.0, 0.0, 1.0], np.float32)
    idx = torch.from_numpy(np.repeat(np.arange(5, dtype=np.int32), 200)).cuda()
    Tt = torch.from_numpy(np.repeat(T, 200)).cuda()
    tok, valid = ms.top_k_top_p_sampling_from_logits(torch.from_numpy(rows).cuda(), Tt, None, 0.9, None, "joint",
                                                     idx, seed=1, offset=0)
    tok, valid = tok.cpu().numpy().reshape(5, 200), valid.cpu().numpy().reshape(5, 200)
    assert valid[0].all() and valid[4].all()
    assert not valid[1].any() and not valid[2].any() and not valid[3].any()
    assert (tok[1:4] == -1).all()
    assert (tok[4] % 2 == 1).all()


def test_long_rows_and_underflow(ms):
    """Rows long enough that a segment spans several blocks (V = 600001: the online
    softmax combines the blocks of a segment), logits far below the maximum (weights
    that underflow to 0) and whole segments of -inf: membership of every draw in both
    orders against the oracle's sets, and the law on the short row."""
    import torch
    rng = np.random.default_rng(2025)
    V = 600_001
    uses = lambda i: [(40, 0.8, None, "top_k_first"), (40, 0.8, None, "joint")]
    Z = _logit_rows(2, V, 3.0, 4242, uses)
    Z[1, :300_000] -= 200.0            # weights exp(-200 - ...) underflow to 0
    Z[1, 400_000:420_000] = -np.inf     # whole segments of -inf
    P = np.stack([filters.softmax(z) for z in Z])
    for i in range(2):
        assert guard_accept(uses)(i, P[i])
    k = np.full(2, 40, np.int32)
    p = np.full(2, 0.8, np.float32)
    Zt = torch.from_numpy(Z).cuda()
    for order in ("top_k_first", "joint"):
        masks, vref = allowed_masks(P, k, p, None, order)
        for call in range(4):
            tok, valid = ms.top_k_top_p_sampling_from_logits(Zt, None, torch.from_numpy(k).cuda(),
                                                             torch.from_numpy(p).cuda(), None, order,
                                                             seed=17, offset=call)
            tok, valid = tok.cpu().numpy(), valid.cpu().numpy()
            assert np.array_equal(valid.astype(bool), vref)
            assert masks[np.arange(2), tok].all(), "a draw outside S"
