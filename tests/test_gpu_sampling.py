"""Parity of the samplers with the oracle.

A sampled token is not unique, so the checks are: every draw lies in the oracle's
allowed set S (exact, on every draw); valid flags are exact; the empirical law of
many draws matches p~ (total variation <= 0.005 with the draw count chosen so the
null expectation is <= 0.002, and a chi-square test at alpha = 1e-3); the round
count respects the halving bound; and, replaying the same Philox stream, the
oracle's step-by-step dual-pivot run lands on the same token except where float32
and float64 prefix sums straddle a boundary.
"""
import numpy as np
import pytest

import workloads
from oracle import dual_pivot, filters, philox
from tests.helpers import (allowed_masks, chi2_pvalue, draws_for_tv, ensure_built, expected_null_tv,
                           guard_accept, tv_distance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ms():
    ensure_built()
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import min_sampling_gb300
    return min_sampling_gb300


def _t(x, dtype):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda()


ENTRIES = ["from_probs", "top_k", "top_p", "min_p", "top_k_first", "joint"]


def _call(ms, entry, probs_t, k, p, mp, indices=None, seed=1, offset=0):
    """Run one entry; k/p/mp are numpy per-output-row arrays (unused ones ignored)."""
    import torch
    idx = None if indices is None else _t(indices, torch.int32)
    kw = dict(seed=seed, offset=offset, return_rounds=True)
    if entry == "from_probs":
        r = ms.sampling_from_probs(probs_t, idx, **kw)
    elif entry == "top_k":
        r = ms.top_k_sampling(probs_t, _t(k, torch.int32), idx, **kw)
    elif entry == "top_p":
        r = ms.top_p_sampling(probs_t, _t(p, torch.float32), idx, **kw)
    elif entry == "min_p":
        r = ms.min_p_sampling(probs_t, _t(mp, torch.float32), idx, **kw)
    else:
        r = ms.top_k_top_p_sampling(probs_t, _t(k, torch.int32), _t(p, torch.float32),
                                    None if mp is None else _t(mp, torch.float32),
                                    order=entry if entry == "joint" else "top_k_first", indices=idx, **kw)
    torch.cuda.synchronize()
    return tuple(x.cpu().numpy() for x in r)


def _oracle_args(entry, k, p, mp):
    """(top_k, top_p, min_p, order) the oracle sees for one entry."""
    if entry == "from_probs":
        return None, None, None, "joint"
    if entry == "top_k":
        return k, None, None, "joint"
    if entry == "top_p":
        return None, p, None, "joint"
    if entry == "min_p":
        return None, None, mp, "joint"
    return k, p, mp, entry


# ------------------------------------------------------------------ Philox

def test_philox_bit_exact(ms):
    import torch
    kat = [((0, 0, 0, 0), (0, 0)), ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2),
           ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0))]
    rng = np.random.default_rng(0)
    ctr = np.concatenate([np.array([c for c, _ in kat], np.uint32),
                          rng.integers(0, 2 ** 32, (5000, 4), dtype=np.uint64).astype(np.uint32)])
    key = np.concatenate([np.array([k for _, k in kat], np.uint32),
                          rng.integers(0, 2 ** 32, (5000, 2), dtype=np.uint64).astype(np.uint32)])
    out = ms.philox4x32_10(_t(ctr.view(np.int32), torch.int32), _t(key.view(np.int32), torch.int32))
    got = out.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, philox.philox4x32_10_np(ctr, key))
    assert tuple(got[0]) == (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)


# ------------------------------------------------------------------ config 1: laws and replay

def _config1():
    params = [(1, 1.0, 0.0), (10, 0.9, 0.0), (50, 0.95, 0.1), (1024, 0.5, 0.0)]

    def uses(i):
        k, p, mp = params[i]
        return [(None, p, None, "joint"), (k, p, mp, "top_k_first"), (k, p, mp, "joint")]
    return workloads.config1(accept=guard_accept(uses))


@pytest.mark.parametrize("entry", ENTRIES)
def test_config1_law(ms, entry):
    """Every draw in S; TV <= 0.005 and chi-square p > 1e-3 per row (config 1)."""
    import torch
    w = _config1()
    P = torch.from_numpy(w.probs).cuda()
    for r in range(4):
        k, p, mp = int(w.top_k[r]), float(w.top_p[r]), float(w.min_p[r])
        ok_args = _oracle_args(entry, k, p, mp)
        pt, ok = filters.filtered_distribution(w.probs[r], *ok_args)
        assert ok
        n = draws_for_tv(pt)
        idx = np.full(n, r, np.int32)
        tok, valid, rounds = _call(ms, entry, P, np.full(n, k, np.int32), np.full(n, p, np.float32),
                                   np.full(n, mp, np.float32), indices=idx, seed=1234 + r, offset=7)
        assert valid.all() and (tok >= 0).all()
        assert (pt[tok] > 0).all(), "a draw outside S"
        counts = np.bincount(tok, minlength=w.vocab).astype(np.float64)
        tv = tv_distance(counts, pt)
        assert tv <= 0.005, (entry, r, tv, expected_null_tv(pt, n))
        assert chi2_pvalue(counts, pt) > 1e-3, (entry, r)
        assert rounds.max() <= filters.round_bound(w.probs[r], *ok_args)


@pytest.mark.parametrize("entry", ENTRIES)
def test_config1_replay_matches_oracle_steps(ms, entry):
    """Same Philox stream: the oracle's float64 run of the pages' algorithm and the
    kernel land on the same token and round count for nearly every draw."""
    import torch
    w = _config1()
    P = torch.from_numpy(w.probs).cuda()
    n_per = 400
    idx = np.repeat(np.arange(4, dtype=np.int32), n_per)
    ks, ps, mps = w.top_k[idx], w.top_p[idx], w.min_p[idx]
    seed, offset = 987654321012345, 2 ** 33 + 5
    tok, valid, rounds = _call(ms, entry, P, ks, ps, mps, indices=idx, seed=seed, offset=offset)
    agree = 0
    for b in range(idx.size):
        r = int(idx[b])
        args = _oracle_args(entry, int(ks[b]), float(ps[b]), float(mps[b]))
        t_ref, ok_ref, r_ref = dual_pivot.sample_philox(w.probs[r], *args, seed=seed, offset=offset, row=b)
        assert bool(valid[b]) == ok_ref
        if t_ref == tok[b] and r_ref == rounds[b]:
            agree += 1
    assert agree >= 0.995 * idx.size, agree


# ------------------------------------------------------------------ full-size configs

def _membership(masks, valid_ref, tok, valid):
    assert np.array_equal(valid.astype(bool), valid_ref)
    ok = valid_ref
    assert (tok[~ok] == -1).all()
    assert masks[np.nonzero(ok)[0], tok[ok]].all(), "a draw outside S"


def test_config3_top_k_first_and_joint(ms):
    """B=64, V=151936, top-k 50 + top-p 0.9: membership on every draw over several calls."""
    import torch
    acc = guard_accept(lambda i: [(50, 0.9, None, "top_k_first"), (50, 0.9, None, "joint")])
    w = workloads.config3(accept=acc, with_logits=False)
    P = torch.from_numpy(w.probs).cuda()
    for order in ("top_k_first", "joint"):
        masks, vref = allowed_masks(w.probs, w.top_k, w.top_p, None, order)
        bounds = [filters.round_bound(w.probs[i], 50, 0.9, None, order) for i in range(64)]
        for call in range(6):
            tok, valid, rounds = _call(ms, order, P, w.top_k, w.top_p, None, seed=42, offset=call)
            _membership(masks, vref, tok, valid)
            assert (rounds <= np.array(bounds)).all()
        # 64 parallel samples of every row through `indices`.
        idx = np.repeat(np.arange(64, dtype=np.int32), 64)
        tok, valid, rounds = _call(ms, order, P, w.top_k[idx], w.top_p[idx], None, indices=idx, seed=3, offset=9)
        _membership(masks[idx], vref[idx], tok, valid)


def test_config2_joint(ms):
    """B=64, V=32000, per-row temperature, k ~ U{1..100}, p ~ U[0.7, 1]: membership on
    every draw; chi-square on four rows at 10^6 draws each."""
    import torch
    w0 = workloads.config2()
    acc = guard_accept(lambda i: [(int(w0.top_k[i]), float(w0.top_p[i]), None, "joint")])
    w = workloads.config2(accept=acc)
    P = torch.from_numpy(w.probs).cuda()
    masks, vref = allowed_masks(w.probs, w.top_k, w.top_p, None, "joint")
    for call in range(4):
        tok, valid, _ = _call(ms, "joint", P, w.top_k, w.top_p, None, seed=100 + call, offset=call)
        _membership(masks, vref, tok, valid)
    for r in (0, 1, 2, 3):
        n = 10 ** 6
        idx = np.full(n, r, np.int32)
        tok, valid, _ = _call(ms, "joint", P, np.full(n, w.top_k[r], np.int32), np.full(n, w.top_p[r], np.float32),
                              None, indices=idx, seed=5, offset=r)
        pt, _ = filters.filtered_distribution(w.probs[r], int(w.top_k[r]), float(w.top_p[r]), None, "joint")
        counts = np.bincount(tok, minlength=w.vocab).astype(np.float64)
        assert (pt[tok] > 0).all()
        assert tv_distance(counts, pt) <= 0.005
        assert chi2_pvalue(counts, pt) > 1e-3


@pytest.mark.parametrize("batch_in", [1, 512])
def test_config4_min_p_and_top_p_parallel_samples(ms, batch_in):
    """V=128256, Student-t logits, 4 outputs per input row: membership, and the four
    parallel samples of a row draw from distinct streams."""
    import torch
    w = workloads.config4(batch_in=batch_in, accept=guard_accept(lambda i: [(None, 0.95, None, "joint")]))
    P = torch.from_numpy(w.probs).cuda()
    check_rows = np.arange(batch_in) if batch_in <= 8 else np.arange(0, batch_in, batch_in // 16)
    sel = np.isin(w.indices, check_rows)
    for entry in ("min_p", "top_p"):
        ref = {}
        for r in check_rows:
            args = (None, None, float(w.min_p[0]), "joint") if entry == "min_p" else (None, float(w.top_p[0]), None, "joint")
            S = filters.allowed_set(w.probs[r], *args)
            m = np.zeros(w.vocab, bool)
            m[S] = True
            ref[int(r)] = m
        seen_distinct = 0
        for call in range(8):
            tok, valid, _ = _call(ms, entry, P, None, w.top_p, w.min_p, indices=w.indices, seed=11, offset=call)
            assert valid.all()
            for b in np.nonzero(sel)[0]:
                assert ref[int(w.indices[b])][tok[b]], (entry, b)
            four = tok.reshape(batch_in, 4)
            seen_distinct += int((four != four[:, :1]).any(axis=1).sum())
        # Rows whose allowed set has several tokens must not repeat one sample 4x every call.
        multi = [r for r in check_rows if ref[int(r)].sum() > 1]
        if multi:
            assert seen_distinct > 0


def test_config5_adversarial_valid_flags_and_rounds(ms):
    """B=256, V=256000: Zipf and near-flat rows, 5% bad rows; joint k=V/2, p=0.99,
    min_p=0.01.  valid = 0 exactly on the bad rows; membership; round bound."""
    import torch
    w = workloads.config5()
    P = torch.from_numpy(w.probs).cuda()
    masks, vref = allowed_masks(w.probs, w.top_k, w.top_p, w.min_p, "joint")
    bad = np.zeros(256, bool)
    bad[w.bad_rows] = True
    assert np.array_equal(~vref, bad)
    bounds = np.array([filters.round_bound(w.probs[i], int(w.top_k[i]), float(w.top_p[i]),
                                           float(w.min_p[i]), "joint") for i in range(256)])
    for call in range(3):
        tok, valid, rounds = _call(ms, "joint", P, w.top_k, w.top_p, w.min_p, seed=77, offset=call)
        _membership(masks, vref, tok, valid)
        assert (rounds[vref] <= bounds[vref]).all()
        assert (rounds[vref] >= 1).all()


# ------------------------------------------------------------------ edge cases

def test_edge_cases(ms):
    import torch
    rng = np.random.default_rng(8)
    for V in (1, 2, 3, 7, 513):
        p = workloads.random_small_rows(1, V, seed=V)[0]
        P = _t(p[None, :], torch.float32)
        n = 2000
        idx = np.zeros(n, np.int32)
        for entry in ENTRIES:
            k, pp, mp = max(1, V // 2), 0.6, 0.2
            tok, valid, _ = _call(ms, entry, P, np.full(n, k, np.int32), np.full(n, pp, np.float32),
                                  np.full(n, mp, np.float32), indices=idx, seed=V, offset=1)
            S = filters.allowed_set(p, *_oracle_args(entry, k, pp, mp))
            assert valid.all() and np.isin(tok, S).all(), (V, entry)
    p = workloads.random_small_rows(1, 50, seed=1)[0]
    P = _t(np.stack([p, p, p, p, p, p]), torch.float32)
    am = int(np.argmax(p))
    k = np.array([1, 50, 0, 3, 3, 3], np.int32)
    tp = np.array([1.0, 0.0, 1.0, np.nan, 0.5, 0.5], np.float32)
    mp = np.array([0.0, 0.0, 1.0, 0.0, 1.5, np.nan], np.float32)
    tok, valid, _ = _call(ms, "joint", P, k, tp, mp, seed=1, offset=2)
    assert tok[0] == am and tok[1] == am and tok[2] == am      # k=1, top_p=0, min_p=1: the arg-max
    assert valid.tolist() == [1, 1, 1, 0, 0, 0] and (tok[3:] == -1).all()
    # Out-of-range indices and bad rows.
    Q = np.stack([p, p, p]).astype(np.float32)
    Q[1, 3] = np.nan
    Q[2, :] = 0
    idx = np.array([0, 1, 2, 3, -1, 0], np.int32)
    tok, valid, _ = _call(ms, "from_probs", _t(Q, torch.float32), None, None, None, indices=idx, seed=3, offset=0)
    assert valid.tolist() == [1, 0, 0, 0, 0, 1] and (tok[1:5] == -1).all()
    # Empty output batch: nothing launched, nothing written.
    out = ms.top_k_sampling(_t(Q, torch.float32), _t(np.zeros(0, np.int32), torch.int32),
                            _t(np.zeros(0, np.int32), torch.int32), seed=0, offset=0)
    assert out[0].numel() == 0


def test_determinism_and_offsets(ms):
    import torch
    w = workloads.config1()
    P = torch.from_numpy(w.probs).cuda()
    n = 4096
    idx = np.repeat(np.arange(4, dtype=np.int32), n // 4)
    args = (w.top_k[idx], w.top_p[idx], w.min_p[idx])
    a = _call(ms, "joint", P, *args, indices=idx, seed=5, offset=10)
    b = _call(ms, "joint", P, *args, indices=idx, seed=5, offset=10)
    c = _call(ms, "joint", P, *args, indices=idx, seed=5, offset=11)
    d = _call(ms, "joint", P, *args, indices=idx, seed=6, offset=10)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[0], c[0]) and not np.array_equal(a[0], d[0])


def test_candidates_concentrated_in_one_cta(ms):
    """Most large values inside the first eighth of the row, so that one CTA holds more
    candidates than its share of the on-chip list (top-k-first prologue, joint
    compaction): membership of every draw."""
    import torch
    Z = workloads.concentrated_logits(2, 151936, 1000, 19000, seed=31)
    P = np.stack([workloads.detie(workloads.softmax_fp32(z))[0] for z in Z])
    acc = guard_accept(lambda i: [(100, 0.9, None, "top_k_first"), (400, 0.95, None, "joint")])
    for i in range(2):
        assert acc(i, P[i]), "the fixed rows sit too close to a top-p boundary"
    Pt = _t(P, torch.float32)
    idx = np.repeat(np.arange(2, dtype=np.int32), 32)
    for entry, k, p in (("top_k_first", 100, 0.9), ("joint", 400, 0.95)):
        ks = np.full(64, k, np.int32)
        ps = np.full(64, p, np.float32)
        masks, vref = allowed_masks(P[idx], ks, ps, None, entry)
        for call in range(4):
            tok, valid, rounds = _call(ms, entry, Pt, ks, ps, None, indices=idx, seed=5, offset=call)
            _membership(masks, vref, tok, valid)


def test_misaligned_rows_and_large_k_first(ms):
    """A base address that is not 16-byte aligned (scalar path) and a top-k-first k
    whose candidates exceed the on-chip list (bisection prologue)."""
    import torch
    acc = guard_accept(lambda i: [(5000, 0.8, None, "top_k_first"), (60, 0.8, None, "top_k_first")])
    w = workloads.config3(batch=8, vocab=40001, accept=acc, with_logits=False)
    flat = torch.empty(w.probs.size + 1, dtype=torch.float32, device="cuda")
    flat[1:] = torch.from_numpy(w.probs.reshape(-1)).cuda()
    P = flat[1:].view(w.probs.shape)
    for k in (60, 5000):
        ks = np.full(8, k, np.int32)
        ps = np.full(8, 0.8, np.float32)
        masks, vref = allowed_masks(w.probs, ks, ps, None, "top_k_first")
        for call in range(3):
            tok, valid, rounds = _call(ms, "top_k_first", P, ks, ps, None, seed=9, offset=call)
            _membership(masks, vref, tok, valid)


def test_misaligned_long_rows_on_the_two_launch_finishes(ms):
    """Scalar loads on the finishing launches: a base address off the 16-byte grid and
    V % 4 != 0, with rows long enough for the joint finish's candidate list and second
    list (not the whole row on chip).  Joint top-k + top-p, min-p (its threshold bounds
    the candidates) and sampling without filters; every draw in S over several calls,
    and 16 parallel samples of every row through `indices`."""
    import torch
    acc = guard_accept(lambda i: [(50, 0.9, None, "joint")])
    w = workloads.config3(batch=8, vocab=100003, accept=acc, with_logits=False)
    flat = torch.empty(w.probs.size + 1, dtype=torch.float32, device="cuda")
    flat[1:] = torch.from_numpy(w.probs.reshape(-1)).cuda()
    P = flat[1:].view(w.probs.shape)
    ks = np.full(8, 50, np.int32)
    ps = np.full(8, 0.9, np.float32)
    mps = np.full(8, 0.1, np.float32)
    cases = [("joint", ks, ps, None), ("min_p", None, None, mps), ("from_probs", None, None, None)]
    for entry, k, p, mp in cases:
        oa = _oracle_args(entry, k, p, mp)
        masks, vref = allowed_masks(w.probs, oa[0], oa[1], oa[2], oa[3])
        for call in range(3):
            tok, valid, rounds = _call(ms, entry, P, k, p, mp, seed=13, offset=call)
            _membership(masks, vref, tok, valid)
        idx = np.repeat(np.arange(8, dtype=np.int32), 16)
        kk = None if k is None else k[idx]
        pp = None if p is None else p[idx]
        mm = None if mp is None else mp[idx]
        tok, valid, _ = _call(ms, entry, P, kk, pp, mm, indices=idx, seed=17, offset=4)
        _membership(masks[idx], vref[idx], tok, valid)


def test_single_pivot_ablation(ms):
    """The one-pivot rule ([blog] rejection sampling) through the ablation entry: the
    same law (TV, chi-square, every draw in S), the oracle's one-pivot run replayed on
    the same Philox stream, and more rounds than the dual-pivot rule where the second
    pivot matters."""
    import torch
    w = _config1()
    P = torch.from_numpy(w.probs).cuda()
    for r in (0, 1):
        k, p = int(w.top_k[r]), float(w.top_p[r])
        pt, ok = filters.filtered_distribution(w.probs[r], k, p, None, "joint")
        n = draws_for_tv(pt)
        idx = torch.from_numpy(np.full(n, r, np.int32)).cuda()
        kk = torch.full((n,), k, dtype=torch.int32, device="cuda")
        pp = torch.full((n,), p, dtype=torch.float32, device="cuda")
        out = {}
        for piv in (1, 2):
            tok, valid, rounds = ms.top_k_top_p_sampling_pivots(P, kk, pp, None, "joint", idx, pivots=piv,
                                                                 seed=99 + r, offset=4, return_rounds=True)
            tok, valid, rounds = tok.cpu().numpy(), valid.cpu().numpy(), rounds.cpu().numpy()
            assert valid.all() and (pt[tok] > 0).all()
            counts = np.bincount(tok, minlength=w.vocab).astype(np.float64)
            assert tv_distance(counts, pt) <= 0.005
            assert chi2_pvalue(counts, pt) > 1e-3
            out[piv] = (tok, rounds)
        # Row 0 keeps the arg-max alone (k = 1): there the second pivot skips most of the
        # rejections (the oracle's one-pivot run averages about 2.6 draws, dual 2.0).
        if r == 0:
            assert out[1][1].mean() > out[2][1].mean() + 0.3
        assert out[1][1].max() >= out[2][1].max()
        agree = 0
        for b in range(400):
            t_ref, _, r_ref = dual_pivot.sample_philox(w.probs[r], k, p, None, "joint", seed=99 + r, offset=4, row=b,
                                                       midpoint="single")
            agree += int(t_ref == out[1][0][b] and r_ref == out[1][1][b])
        assert agree >= 0.99 * 400, agree
    with pytest.raises(ms.FsError):
        ms.top_k_top_p_sampling_pivots(P, 10, 0.9, None, "joint", pivots=3, seed=1, offset=0)


def test_refined_bound_and_long_list_law(ms):
    """Top-k-first draws where the top-k bound is refined inside its histogram bin
    (a near-flat row, k = 50) and where the candidate list is longer than the
    register path (an N(0, 3^2) softmax row, k = 300, top-p 0.95): every draw in S,
    TV <= 0.005 and chi-square p > 1e-3 against the oracle's filtered law."""
    import torch
    V = 151936
    rng = np.random.default_rng([17, V])
    flat = workloads.detie(workloads.softmax_fp32(rng.normal(0, 0.05, V)))[0]
    acc = guard_accept(lambda i: [(300, 0.95, None, "top_k_first")])
    steep = None
    for att in range(64):
        cand = workloads.detie(workloads.softmax_fp32(workloads.row_rng(18, 0, att).normal(0, 3, V)))[0]
        if acc(0, cand):
            steep = cand
            break
    assert steep is not None
    P = np.stack([flat, steep])
    Pt = _t(P, torch.float32)
    for r, (k, p) in enumerate([(50, 1.0), (300, 0.95)]):
        pt, ok = filters.filtered_distribution(P[r], k, p, None, "top_k_first")
        assert ok
        n = draws_for_tv(pt)
        idx = np.full(n, r, np.int32)
        tok, valid, rounds = _call(ms, "top_k_first", Pt, np.full(n, k, np.int32), np.full(n, p, np.float32),
                                   None, indices=idx, seed=4321 + r, offset=3)
        assert valid.all() and (tok >= 0).all()
        assert (pt[tok] > 0).all(), "a draw outside S"
        counts = np.bincount(tok, minlength=V).astype(np.float64)
        tv = tv_distance(counts, pt)
        assert tv <= 0.005, (r, tv, expected_null_tv(pt, n))
        assert chi2_pvalue(counts, pt) > 1e-3, r


@pytest.mark.parametrize("V", [32000, 151936, 256000])
def test_launch_plan_fits_one_wave(ms, V):
    """The launch plans of both kinds.  Top-k-first (scan, then one CTA per row): one
    CTA covers the whole row's summary.  Joint (rejection rounds on a cluster): a
    cluster of 1..16 CTAs covering the row's segments, at most the occupancy limit of
    CTAs per SM, every cluster resident at once whenever C > 1 (rows x C <= SMs x CTAs
    per SM)."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for B in (1, 8, 32, 64, 128, 192, 256, 4096):
        pl = ms.sampling_plan(B, V, "top_k_first")
        assert pl["cluster"] == 1 and 1 <= pl["ctas_per_sm"] <= 8, pl
        assert pl["segments_per_cta"] * pl["segment_len"] >= V > (pl["segments_per_cta"] - 1) * pl["segment_len"]
        pl = ms.sampling_plan(B, V, "joint")
        C, per_sm = pl["cluster"], pl["ctas_per_sm"]
        assert 1 <= C <= 16 and 1 <= per_sm <= 8, pl
        assert C * pl["segments_per_cta"] * pl["segment_len"] >= V, pl
        assert pl["segments_per_cta"] % 4 == 0
        if C > 1:
            assert B * C <= sms * per_sm, (B, pl)
        for order in ("top_k_first", "joint"):
            assert ms.sampling_plan(B, V, order) == ms.sampling_plan(B, V, order)   # cached, stable
    with pytest.raises(ValueError):
        ms.sampling_plan(8, V, "sorted")


def test_batch_sizes_and_cluster_sizes(ms):
    """Batch sizes whose launch plans use clusters of many sizes (16 down to 2 CTAs per
    row, odd sizes included), V = 32000: membership of every draw in both orders (the
    joint order on those clusters), top-k / top-p renormalisation and the logit mask
    exactly as the oracle's."""
    import torch
    from tests.test_gpu_filters import _check_renorm, _run as run_filter
    V = 32000
    seen = set()
    for B in (3, 33, 45, 60, 77, 100, 130, 300):
        acc = guard_accept(lambda i: [(50, 0.9, None, "top_k_first"), (None, 0.9, None, "joint"),
                                      (50, 0.9, None, "joint")])
        w = workloads.config3(batch=B, vocab=V, accept=acc, seed=9000 + B)
        seen.add(ms.sampling_plan(B, V, "joint")["cluster"])
        P = torch.from_numpy(w.probs).cuda()
        ks = np.full(B, 50, np.int32)
        ps = np.full(B, 0.9, np.float32)
        for order in ("top_k_first", "joint"):
            masks, vref = allowed_masks(w.probs, ks, ps, None, order)
            for call in range(2):
                tok, valid, rounds = _call(ms, order, P, ks, ps, None, seed=B, offset=call)
                _membership(masks, vref, tok, valid)
        out, valid = run_filter(ms, "top_k", w.probs, list(ks))
        _check_renorm(w.probs, list(ks), out, valid, filters.top_k_renorm)
        out, valid = run_filter(ms, "top_p", w.probs, list(ps))
        _check_renorm(w.probs, list(ps), out, valid, filters.top_p_renorm)
        out, valid = run_filter(ms, "mask", w.logits, list(ks))
        for i in range(B):
            exp, ok = filters.top_k_mask_logits(w.logits[i], 50)
            assert ok and valid[i] and np.array_equal(out[i], exp), (B, i)
    assert len(seen) >= 5, seen
