"""Pins of the CPU oracle to facts that do not come from the oracle itself.

* the pages' worked rows (tests/golden/hand_rows.json, each with its citation);
* the closed form of the correctness theorem, Pr[out = j] = p_j / Z, checked
  exactly (rational arithmetic) against the dual-pivot algorithm's own recurrence;
* brute-force membership by counting (no sort) against the sort-based sets;
* Philox4x32-10 known-answer vectors of its published reference implementation;
* special cases with textbook answers (k = 1 is arg-max, k = V is no filter,
  top-p 1 keeps every positive entry, min-p 1 keeps the maximum, ...);
* planted mistakes in the oracle that these pins must catch.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import bruteforce, dual_pivot, filters, philox
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_rows.json")


def _cases():
    with open(GOLDEN) as fh:
        return json.load(fh)["cases"]


def _ratio(s: str) -> float:
    a, b = s.split("/")
    return float(a) / float(b)


# ---------------------------------------------------------------- hand rows

@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["id"])
def test_hand_row_sets_and_values(case):
    p = np.array(case["probs"], np.float32)
    args = (case["top_k"], case["top_p"], case["min_p"], case["order"])
    S = filters.allowed_set(p, *args)
    assert S.tolist() == case["expected_set"]
    assert bruteforce.members(p, *args).tolist() == case["expected_set"]
    pt, ok = filters.filtered_distribution(p, *args)
    assert ok
    for j, r in case["expected_ptilde"].items():
        assert abs(pt[int(j)] - _ratio(r)) < 1e-6
    assert abs(pt.sum() - 1.0) < 1e-12
    law = dual_pivot.exact_output_law(p, *args)
    assert sorted(law) == case["expected_set"]
    for j, r in case["expected_ptilde"].items():
        assert abs(float(law[int(j)]) - _ratio(r)) < 1e-6


def test_drill_threshold_and_prefix_masses():
    c = _cases()[0]
    p = np.array(c["probs"], np.float32)
    assert filters.top_p_threshold(p, c["top_p"]) == pytest.approx(np.float32(c["expected_threshold"]), abs=0)
    vals = np.sort(p.astype(np.float64))[::-1]
    assert np.allclose(np.cumsum(vals)[:3], c["expected_prefix_masses"], atol=1e-7)
    c2 = _cases()[1]
    assert filters.top_k_threshold(p, c2["top_k"]) == np.float32(c2["expected_threshold"])
    out, ok = filters.top_p_renorm(p, 0.8)
    assert ok and np.allclose(out, [0, 0.40 / 0.85, 0, 0.30 / 0.85, 0.15 / 0.85], atol=1e-7)
    out, ok = filters.top_k_renorm(p, 2)
    assert ok and np.allclose(out, [0, 0.40 / 0.70, 0, 0.30 / 0.70, 0], atol=1e-7)


def test_explainer_topk_walkthrough_rounds():
    """The explainer's walk-through: drawing D then C raises `low` to 0.12 then 0.18,
    after which only A and B remain and every further draw is accepted."""
    p = np.array([0.35, 0.28, 0.18, 0.12, 0.07], np.float32)
    row = dual_pivot._Row(p, 2, None, None, "joint")
    assert not row.f(np.float32(0.12)) and not row.f(np.float32(0.18))
    assert row.f(np.float32(0.28)) and row.f(np.float32(0.35))
    # From low = 0.18 only A and B are drawable; both are accepted.
    for u in (0.0, 0.3, 0.6, 0.99):
        j = dual_pivot.draw_inverse_transform(p.astype(np.float64), float(np.float32(0.18)), u)
        assert j in (0, 1)


# ---------------------------------------------------------------- brute force vs sort

EDGE_K = [None, 0, 1, 2, 3, 5, 7, 8, 9]
EDGE_P = [None, 0.0, 1e-3, 0.3, 0.5, 0.75, 0.9, 0.999, 1.0]
EDGE_MINP = [None, 0.0, 0.05, 0.3, 0.7, 1.0, 1.5]


def test_bruteforce_matches_sorted_sets():
    rng = np.random.default_rng(5)
    n_checked = 0
    for V in (1, 2, 3, 5, 8):
        rows = workloads.random_small_rows(60, V, seed=100 + V, zero_prob=0.2)
        for p in rows:
            if not (p > 0).any():
                continue
            for order in filters.ORDERS:
                for _ in range(12):
                    k = EDGE_K[rng.integers(len(EDGE_K))]
                    tp = EDGE_P[rng.integers(len(EDGE_P))]
                    mp = EDGE_MINP[rng.integers(len(EDGE_MINP))]
                    if filters.topp_boundary_margin(p, k, tp, mp, order) < 1e-9:
                        continue
                    a = filters.allowed_set(p, k, tp, mp, order).tolist()
                    b = bruteforce.members(p, k, tp, mp, order).tolist()
                    assert a == b, (p, k, tp, mp, order)
                    n_checked += 1
    assert n_checked > 3000


# ---------------------------------------------------------------- closed form of the theorem

def _closed_form(p, k, tp, mp, order):
    S = filters.allowed_set(p, k, tp, mp, order)
    vals = {int(j): Fraction(float(np.float32(p[j]))) for j in S}
    Z = sum(vals.values(), Fraction(0))
    return {j: v / Z for j, v in vals.items()}


@pytest.mark.parametrize("midpoint", ["exact", "fp32"])
def test_exact_law_equals_pj_over_Z(midpoint):
    rng = np.random.default_rng(7 if midpoint == "exact" else 8)
    n = 0
    for V in (1, 2, 3, 4, 5, 6):
        rows = workloads.random_small_rows(8, V, seed=300 + V, zero_prob=0.15)
        for p in rows:
            if not (p > 0).any():
                continue
            for order in filters.ORDERS:
                for _ in range(4):
                    k = EDGE_K[rng.integers(len(EDGE_K))]
                    tp = EDGE_P[rng.integers(len(EDGE_P))]
                    mp = EDGE_MINP[rng.integers(len(EDGE_MINP))]
                    if filters.topp_boundary_margin(p, k, tp, mp, order) < 1e-9:
                        continue
                    law = dual_pivot.exact_output_law(p, k, tp, mp, order, midpoint=midpoint)
                    assert law == _closed_form(p, k, tp, mp, order), (p, k, tp, mp, order)
                    n += 1
    assert n > 150


def test_single_pivot_law_is_exact_and_never_faster():
    """The one-pivot sampler of the [blog] rejection-sampling section is also exact
    (p_j / Z on S), and on a row where the dual-pivot rule skips several rejections its
    expected number of draws is larger."""
    p = np.array([0.02, 0.03, 0.05, 0.10, 0.15, 0.20, 0.45], np.float32)
    for k, tp in [(1, None), (2, None), (None, 0.5), (3, 0.9)]:
        law = dual_pivot.exact_output_law(p, k, tp, None, "joint", midpoint="single")
        S = filters.allowed_set(p, k, tp, None, "joint")
        Z = sum(Fraction(float(p[i])) for i in S)
        assert set(law) == set(int(i) for i in S)
        for i in S:
            assert law[int(i)] == Fraction(float(p[i])) / Z
    # Expected draws from the start state, by the same recursion with a draw counter.
    def expected_draws(midpoint):
        row = dual_pivot._Row(p, 1, None, None, "joint", exact=True)

        def go(low, high):
            elig = [i for i in range(row.V) if row.p[i] > low]
            S_ = sum((row.p[i] for i in elig), Fraction(0))
            e = Fraction(1)
            for i in elig:
                nxt = dual_pivot.three_cases(row, row.p[i], high, midpoint)
                if nxt is not None:
                    e += row.p[i] / S_ * go(*nxt)
            return e
        return go(row.low0, row.high0)
    assert expected_draws("single") > expected_draws("exact")


def test_softmax_definition():
    """Shift invariance, the uniform row, the ratio exp((z_i - z_j) / T), T = 1 against
    a hand value, and weight 0 for -inf."""
    z = np.array([0.0, 1.0, -2.0, 3.5], np.float32)
    for T in (0.5, 1.0, 2.0):
        p = filters.softmax(z, T)
        assert abs(p.sum() - 1.0) < 1e-15
        np.testing.assert_allclose(filters.softmax(z + np.float32(7.0), T), p, rtol=1e-13)
        assert math.isclose(p[1] / p[0], math.exp(1.0 / T), rel_tol=1e-13)
    np.testing.assert_allclose(filters.softmax(np.zeros(5, np.float32)), np.full(5, 0.2), rtol=1e-15)
    q = filters.softmax(np.array([0.0, math.log(3.0)], np.float32))
    assert math.isclose(q[1], 0.75, rel_tol=1e-7)          # e^{ln 3} / (1 + e^{ln 3}) with z rounded to float32
    r = filters.softmax(np.array([1.0, -np.inf, 1.0], np.float32))
    assert r[1] == 0.0 and r[0] == r[2] == 0.5


def test_exact_law_on_an_8_token_row_every_k():
    p = workloads.random_small_rows(1, 8, seed=4242)[0]
    for k in range(1, 9):
        law = dual_pivot.exact_output_law(p, k, None, None)
        assert law == _closed_form(p, k, None, None, "joint")
        assert sum(law.values()) == 1


# ---------------------------------------------------------------- special cases

def test_special_cases():
    p = workloads.random_small_rows(1, 7, seed=9)[0]
    am = int(np.argmax(p))
    pos = np.nonzero(p > 0)[0].tolist()
    assert filters.allowed_set(p, 1).tolist() == [am]                      # k = 1 is greedy
    assert filters.allowed_set(p, 7).tolist() == pos                       # k = V: no filter
    assert filters.allowed_set(p, 0).tolist() == pos                       # k <= 0: no filter
    assert filters.allowed_set(p, None, 1.0).tolist() == pos               # top-p 1 keeps all
    assert filters.allowed_set(p, None, 0.0).tolist() == [am]              # top-p 0: arg-max
    assert filters.allowed_set(p, None, None, 1.0).tolist() == [am]        # min-p 1: the max
    assert filters.allowed_set(p, None, None, 1.5).tolist() == []          # min-p > 1: empty
    pt, ok = filters.filtered_distribution(p)
    assert ok and np.allclose(pt, p / p.astype(np.float64).sum())
    # min-p is invariant to scaling the row (max and threshold scale together).
    assert filters.allowed_set(p * 3, None, None, 0.3).tolist() == filters.allowed_set(p, None, None, 0.3).tolist()


@pytest.mark.parametrize("bad", ["nan", "neg", "zero"])
def test_invalid_rows(bad):
    p = np.array([0.1, 0.2, 0.3, 0.4], np.float32)
    if bad == "nan":
        p[2] = np.nan
    elif bad == "neg":
        p[1] = -0.1
    else:
        p[:] = 0
    assert filters.allowed_set(p, 2, 0.9).size == 0
    assert bruteforce.members(p, 2, 0.9).size == 0
    assert dual_pivot.sample(p, 2, 0.9, uniform=lambda r: 0.5) == (-1, False, 0)
    assert dual_pivot.exact_output_law(p, 2, 0.9) == {}
    out, ok = filters.top_k_renorm(p, 2)
    assert not ok and not out.any()


def test_renorm_and_mask_definitions():
    rng = np.random.default_rng(3)
    for _ in range(50):
        V = int(rng.integers(2, 40))
        p = workloads.random_small_rows(1, V, seed=int(rng.integers(1 << 30)))[0]
        k = int(rng.integers(1, V))
        out, ok = filters.top_k_renorm(p, k)
        assert ok and np.count_nonzero(out) == k and abs(out.sum() - 1) < 1e-12
        kept = out > 0
        assert p[kept].min() > p[~kept].max()
        tp = float(rng.uniform(0.05, 0.95))
        out, ok = filters.top_p_renorm(p, tp)
        kept = np.sort(p[out > 0].astype(np.float64))
        M = p.astype(np.float64).sum()
        assert kept.sum() >= np.float32(tp) * M                  # reaches p
        assert kept[1:].sum() < np.float32(tp) * M               # and is the smallest such prefix
        z = (rng.normal(size=V) * 3).astype(np.float32)
        mz, ok = filters.top_k_mask_logits(z, k)
        assert ok and np.isfinite(mz).sum() == k
        assert set(np.nonzero(np.isfinite(mz))[0]) == set(np.argsort(-z)[:k])
    z = np.array([1.0, np.nan, 2.0], np.float32)
    mz, ok = filters.top_k_mask_logits(z, 1)
    assert not ok and np.isneginf(mz).all()


# ---------------------------------------------------------------- Philox

# Known-answer vectors of the Random123 reference distribution (counter, key, output).
PHILOX_KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,out", PHILOX_KAT)
def test_philox_known_answers(ctr, key, out):
    assert philox.philox4x32_10(ctr, key) == out
    got = philox.philox4x32_10_np(np.array([ctr], np.uint32), np.array([key], np.uint32))
    assert tuple(int(x) for x in got[0]) == out


def test_philox_uniform_grid_and_spread():
    us = np.array([philox.sampler_uniform(123, 7, b, r) for b in range(200) for r in range(20)])
    assert ((us >= 0) & (us < 1)).all()
    assert np.all(us * 2 ** 24 == np.floor(us * 2 ** 24))
    hist = np.histogram(us, bins=10, range=(0, 1))[0]
    assert hist.min() > 300 and hist.max() < 500
    # Different offsets (calls) and rows give different streams.
    assert philox.sampler_uniform(1, 0, 0, 0) != philox.sampler_uniform(1, 1, 0, 0)
    assert philox.sampler_uniform(1, 0, 0, 0) != philox.sampler_uniform(1, 0, 1, 0)


# ---------------------------------------------------------------- replayed sampler

def test_replayed_sampler_matches_law_and_round_bound():
    p = workloads.random_small_rows(1, 16, seed=77)[0]
    for k, tp, mp, order in [(5, None, None, "joint"), (8, 0.6, None, "top_k_first"),
                             (None, 0.7, None, "joint"), (None, None, 0.3, "joint"),
                             (12, 0.8, 0.1, "joint")]:
        pt, _ = filters.filtered_distribution(p, k, tp, mp, order)
        bound = filters.round_bound(p, k, tp, mp, order)
        n = 6000
        counts = np.zeros(16)
        for b in range(n):
            tok, ok, rounds = dual_pivot.sample_philox(p, k, tp, mp, order, seed=99, offset=3, row=b)
            assert ok and pt[tok] > 0 and 1 <= rounds <= bound
            counts[tok] += 1
        tv = 0.5 * np.abs(counts / n - pt).sum()
        assert tv < 0.03


# ---------------------------------------------------------------- planted mistakes

def _law_ok(p, args):
    return dual_pivot.exact_output_law(p, *args) == _closed_form(p, *args)


def test_pins_catch_planted_mistakes(monkeypatch):
    """Each mutation of the oracle below is a plausible slip; a pin must fail on it."""
    # A graded row, so that every case of the three-way update is reached.
    p = np.array([0.30, 0.25, 0.20, 0.15, 0.10], np.float32)
    cases = [(3, None, None, "joint"), (None, 0.6, None, "joint"), (4, 0.7, None, "top_k_first")]
    assert all(_law_ok(p, c) for c in cases)
    orig_f = dual_pivot._Row.f

    def inclusive_mass(self, tau):          # top-p test counting the pivot's own mass
        cnt, mass = self.count_mass_above(tau)
        mass = mass + (Fraction(float(tau)) if self.exact else float(tau))
        if self.k_on and not cnt < self.k:
            return False
        if self.p_on and not (cnt == 0 or mass < self.top_p * self.Mp):
            return False
        return True

    def count_le(self, tau):                # top-k test with <= k
        cnt, mass = self.count_mass_above(tau)
        if self.k_on and not cnt <= self.k:
            return False
        return orig_f(self, tau) or (self.k_on and cnt == self.k)

    for bad in (inclusive_mass, count_le):
        monkeypatch.setattr(dual_pivot._Row, "f", bad)
        assert not all(_law_ok(p, c) for c in cases), bad.__name__
    monkeypatch.setattr(dual_pivot._Row, "f", orig_f)

    # Swapped cases 2 and 3: `low` jumps to pivot2 although f(pivot2) = 1.
    def swapped(row, pivot1, high, midpoint):
        if row.f(pivot1):
            return None
        pivot2 = row.midpoint(pivot1, high, midpoint)
        return (pivot2, high) if row.f(pivot2) else (pivot1, pivot2)

    monkeypatch.setattr(dual_pivot, "three_cases", swapped)
    assert not all(_law_ok(p, c) for c in cases)
    monkeypatch.undo()
    assert all(_law_ok(p, c) for c in cases)

    # The order matters (explainer, filter-order section): on its row with top-p 0.75,
    # top-k-first measures 0.75 * F_k = 0.675 and stops at {A,B} (0.70), while joint
    # measures 0.75 * M = 0.75 and needs {A,B,C}.  Measuring top-k-first against M
    # (a plausible slip) would make the two agree.
    q = np.array([0.40, 0.30, 0.20, 0.10], np.float32)
    assert filters.allowed_set(q, 3, 0.6, None, "top_k_first").tolist() == [0, 1]
    assert filters.allowed_set(q, 3, 0.9, None, "top_k_first").tolist() == [0, 1, 2]
    assert filters.allowed_set(q, 3, 0.9, None, "joint").tolist() == [0, 1, 2]
    assert filters.allowed_set(q, 3, 0.75, None, "top_k_first").tolist() == [0, 1]
    assert filters.allowed_set(q, 3, 0.75, None, "joint").tolist() == [0, 1, 2]
    assert bruteforce.members(q, 3, 0.75, None, "top_k_first").tolist() == [0, 1]
    assert bruteforce.members(q, 3, 0.75, None, "joint").tolist() == [0, 1, 2]


# ---------------------------------------------------------------- generators

def test_generators_tie_free_and_deterministic():
    w = workloads.config1()
    assert w.probs.shape == (4, 1024) and w.probs.dtype == np.float32
    for r in w.probs:
        assert not workloads.has_positive_ties(r)
    w2 = workloads.config1()
    assert np.array_equal(w.probs, w2.probs)
    x, nb = workloads.detie(np.array([0.5, 0.5, 0.5, 0.0, 0.0, 0.25], np.float32))
    assert nb == 2 and not workloads.has_positive_ties(x) and (x == 0).sum() == 2
    w4 = workloads.config4(batch_in=2, vocab=4096)
    assert w4.indices.tolist() == [0, 0, 0, 0, 1, 1, 1, 1]
    w5 = workloads.config5(batch=40, vocab=2000)
    assert len(w5.bad_rows) == 2
    for r in w5.bad_rows:
        assert not filters.row_is_valid(w5.probs[r])


# ---------------------------------------------------------------- round bound and cut value

def _small_cases(seed, n_rows=24):
    """(p, k, top_p, min_p, order) over small rows and parameter edges, skipping rows
    whose top-p boundary is too close to call."""
    rng = np.random.default_rng(seed)
    out = []
    for V in (2, 3, 4, 5, 6, 7, 8):
        for p in workloads.random_small_rows(n_rows, V, seed=seed + V, zero_prob=0.1):
            if not (p > 0).any():
                continue
            for order in filters.ORDERS:
                for _ in range(3):
                    k = EDGE_K[rng.integers(len(EDGE_K))]
                    tp = EDGE_P[rng.integers(len(EDGE_P))]
                    mp = EDGE_MINP[rng.integers(len(EDGE_MINP))]
                    if filters.topp_boundary_margin(p, k, tp, mp, order) < 1e-9:
                        continue
                    out.append((p, k, tp, mp, order))
    return out


_ROUND_CASES = None


def _round_cases():
    """Every case with its longest run of the sampler (the algorithm's own state walk,
    exact rationals, float32 midpoints as the kernels compute them)."""
    global _ROUND_CASES
    if _ROUND_CASES is None:
        _ROUND_CASES = [(c, dual_pivot.max_draws(*c)) for c in _small_cases(900)]
    return _ROUND_CASES


def _geometric_row():
    return np.array([2.0 ** -i for i in range(1, 9)], np.float32)   # 1/2, 1/4, ..., 1/256


def _near_flat_row():
    return np.array([0.26, 0.25, 0.24, 0.23], np.float32)


def _bound_pins_hold(bound) -> bool:
    """The pins of the round bound, for a candidate `bound(p, k, top_p, min_p, order)`.

    1. No run of the algorithm is longer than the bound ([blog] dual pivot: the bound
       is a property of every path, so the longest path of the exact state walk must
       respect it), on every small case.
    2. Two rows worked by hand, one for each of the two limits.
       Geometric row 1/2, 1/4, ..., 1/256 with k = 1: S = {1/2}; seven tokens can be
       rejected, so the count limit is 7 + 1 = 8; tau* = 1/2, a = 1/4, high0 = 1/2,
       log2(high0 / (tau* - a)) = 1, so the halving limit is 3 + 1 = 4.  The bound
       is 4.  (Every run takes at most 2 draws: a rejected draw p_j <= 1/4 puts the
       midpoint (p_j + 1/2) / 2 above 1/4, where f is still false, so `low` jumps past
       every token but 1/2.)
       Near-flat row .26, .25, .24, .23 with k = 1: three tokens can be rejected, so
       the count limit is 4; tau* - a = .01, log2(.26 / .01) = 4.7, so the halving
       limit is 3 + 5 = 8.  The bound is 4.
    """
    for c, longest in _round_cases():
        if longest > bound(*c):
            return False
    return bound(_geometric_row(), 1, None, None, "joint") == 4 and \
        bound(_near_flat_row(), 1, None, None, "joint") == 4


def test_round_bound_covers_every_path_and_hand_rows():
    assert len(_round_cases()) > 1000
    assert _bound_pins_hold(filters.round_bound)
    assert filters.round_bound_terms(_geometric_row(), 1) == (8, 4)
    assert filters.round_bound_terms(_near_flat_row(), 1) == (4, 8)
    assert dual_pivot.max_draws(_geometric_row(), 1) == 2
    assert dual_pivot.max_draws(_near_flat_row(), 1) == 3
    # The bound is not vacuous: on some cases a run reaches it.
    assert any(longest == filters.round_bound(*c) and longest > 1 for c, longest in _round_cases())


def test_round_bound_pins_catch_planted_mistakes():
    """Plausible slips in the bound, each of which a pin must catch."""
    def terms(*c):
        return filters.round_bound_terms(*c) or (0, 0)

    mutants = {
        "max for min": lambda *c: max(terms(*c)),
        "halving limit without the +3": lambda *c: min(terms(*c)[0], terms(*c)[1] - 3),
        "count limit without the +1": lambda *c: min(terms(*c)[0] - 1, terms(*c)[1]),
        "count limit alone, off by one": lambda *c: terms(*c)[0] - 1,
    }
    for name, bad in mutants.items():
        assert not _bound_pins_hold(bad), name


def _f_switches_at(c, cut_fn) -> bool:
    """f(tau) holds at tau = cut and fails at the next float64 below it ([blog]
    rejection sampling: the test is monotone in tau, so the cut is where it turns on)."""
    p, k, tp, mp, order = c
    if filters.allowed_set(p, k, tp, mp, order).size == 0:
        return True
    row = dual_pivot._Row(p, k, tp, mp, order, exact=False)
    cut = cut_fn(p, k, tp, mp, order)
    if not row.f(cut):
        return False
    return cut <= 0.0 or not row.f(np.nextafter(cut, -np.inf))


def test_cut_value_is_where_the_acceptance_test_turns_on():
    cases = _small_cases(950, n_rows=16)
    assert len(cases) > 600
    assert all(_f_switches_at(c, filters.cut_value) for c in cases)
    # Planted mistakes: the smallest active cut instead of the largest; the top-p cut
    # one rank too deep.
    orig = filters.cut_value

    def smallest_cut(p, k, tp, mp, order):
        one = [orig(p, k, None, None, order), orig(p, None, tp, None, order), orig(p, None, None, mp, order)]
        on = [x for x in one if x > 0]
        return min(on) if on else 0.0

    def topp_one_deeper(p, k, tp, mp, order):
        v = orig(p, k, tp, mp, order)
        if tp is None or not (0 < float(np.float32(tp)) < 1):
            return v
        vals = np.sort(p.astype(np.float64)[p > 0])[::-1]
        below = vals[vals < v]
        return float(below[0]) if below.size and v == orig(p, None, tp, None, order) else v

    for bad in (smallest_cut, topp_one_deeper):
        assert not all(_f_switches_at(c, bad) for c in cases), bad.__name__
