"""Pins of the chain speculative-sampling oracle (oracle/speculative.py) to facts
that do not come from the oracle itself:

* the theorem of the method (Leviathan et al. 2023, Appendix A.1): the token
  emitted at a position is distributed exactly as the target row there;
* the law of the accepted count, by enumeration of every draft sequence against
  the product of the per-position acceptance probabilities sum_x min(p, q);
* a Monte Carlo run of the step-by-step ``verify`` against both;
* a hand-worked row and the special cases (q = p always accepts, p(d) = 0 always
  rejects, an out-of-range draft token is rejected);
* a planted mistake (the residual taken the wrong way round) that the theorem pin
  must catch.
"""
import numpy as np
import pytest

from oracle import speculative as spec
from tests.helpers import chi2_pvalue


def _rows(rng, n, V):
    x = rng.dirichlet(np.full(V, 0.7), size=n).astype(np.float32)
    return x / x.sum(axis=1, keepdims=True, dtype=np.float64).astype(np.float32)


@pytest.mark.parametrize("seed", range(5))
def test_first_emission_is_the_target(seed):
    rng = np.random.default_rng(seed)
    p, q = _rows(rng, 2, 7)
    p64 = p.astype(np.float64)
    law = spec.first_emission_law(p, q)
    assert np.allclose(law, p64 / p64.sum(), atol=1e-7)   # float32 rows sum to 1 within 1e-7
    assert abs(law.sum() - 1.0) < 1e-7


def test_planted_residual_mistake_is_caught(monkeypatch):
    rng = np.random.default_rng(11)
    p, q = _rows(rng, 2, 7)
    monkeypatch.setattr(spec, "residual_weights",
                        lambda a, b: np.maximum(spec.as64(b) - spec.as64(a), 0.0))
    law = spec.first_emission_law(p, q)
    assert not np.allclose(law, p.astype(np.float64), atol=1e-3)


@pytest.mark.parametrize("seed", range(3))
def test_accepted_count_law_closed_form(seed):
    rng = np.random.default_rng(100 + seed)
    L, V = 3, 5
    q = _rows(rng, L, V)
    p = _rows(rng, L + 1, V)
    law = spec.accepted_count_law(q, p)
    beta = [sum(min(float(a), float(b)) for a, b in zip(p[i].astype(np.float64), q[i].astype(np.float64)
                                                        / q[i].astype(np.float64).sum()))
            for i in range(L)]
    closed = [np.prod(beta[:i]) * (1 - beta[i]) for i in range(L)] + [np.prod(beta)]
    assert np.allclose(law, closed, atol=1e-9)
    assert np.allclose([spec.acceptance_probability(p[i], q[i]) for i in range(L)], beta, atol=1e-9)


def test_verify_monte_carlo():
    """verify itself, with draft tokens drawn from q and uniform tests: the first
    emitted token follows p_1 and the accepted count follows the enumerated law."""
    rng = np.random.default_rng(7)
    L, V, n = 2, 5, 60_000
    q = _rows(rng, L, V)
    p = _rows(rng, L + 1, V)
    qn = q.astype(np.float64) / q.astype(np.float64).sum(axis=1, keepdims=True)
    first = np.zeros(V)
    acc = np.zeros(L + 1)
    for _ in range(n):
        d = [rng.choice(V, p=qn[i]) for i in range(L)]
        u = rng.random(L + 1)
        toks, a, e = spec.verify(q, d, p, u[:L], u[L])
        assert e == a + 1 and (toks[:a] == d[:a]).all() and toks[a] >= 0 and (toks[a + 1:] == -1).all()
        first[toks[0]] += 1
        acc[a] += 1
    p1 = p[0].astype(np.float64) / p[0].astype(np.float64).sum()
    assert chi2_pvalue(first, p1) > 1e-4
    assert chi2_pvalue(acc, spec.accepted_count_law(q, p)) > 1e-4


def test_hand_worked_row():
    # p1 = (0.2, 0.5, 0.3), q1 = (0.6, 0.3, 0.1), draft d1 = 0: p/q = 1/3.
    q = np.array([[0.6, 0.3, 0.1]], np.float32)
    p = np.array([[0.2, 0.5, 0.3], [0.1, 0.1, 0.8]], np.float32)
    # u = 0.5: 0.5 * 0.6 = 0.3 is not below 0.2, rejected.  Residual max(p - q, 0) =
    # (0, 0.2, 0.2); u_final = 0.25 targets 0.1 of 0.4, reached at index 1.
    toks, a, e = spec.verify(q, [0], p, [0.5], 0.25)
    assert list(toks) == [1, -1] and a == 0 and e == 1
    # u = 0.25: 0.15 < 0.2, accepted; the bonus draw over p2 targets 0.25 of 1.0:
    # running sums 0.1, 0.2, 1.0, reached at index 2.
    toks, a, e = spec.verify(q, [0], p, [0.25], 0.25)
    assert list(toks) == [0, 2] and a == 1 and e == 2


def test_special_cases():
    rng = np.random.default_rng(3)
    q = _rows(rng, 3, 6)
    p = np.concatenate([q, _rows(rng, 1, 6)])
    d = [int(np.argmax(q[i])) for i in range(3)]
    toks, a, e = spec.verify(q, d, p, [0.999999] * 3, 0.5)       # q = p: always accepted
    assert a == 3 and e == 4 and list(toks[:3]) == d
    p0 = p.copy()
    p0[0] = _rows(rng, 1, 6)[0]
    p0[0, d[0]] = 0.0                                            # another target row, zero at d
    toks, a, e = spec.verify(q, d, p0, [0.0] * 3, 0.5)           # p(d) = 0: rejected even at u = 0
    assert a == 0 and e == 1 and toks[0] != d[0] and toks[0] >= 0
    toks, a, e = spec.verify(q, [6, 0, 0], p, [0.0] * 3, 0.5)    # out-of-range draft token
    assert a == 0
    # A residual with no mass (draft and target rows equal at the rejected position,
    # forced by an out-of-range token): nothing is emitted.
    toks, a, e = spec.verify(q, [-1, 0, 0], p, [0.0] * 3, 0.5)
    assert a == 0 and e == 0 and (toks == -1).all()
