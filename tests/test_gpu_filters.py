"""Parity of the filter-only kernels (top_k_renorm_probs, top_p_renorm_probs,
top_k_mask_logits) with the oracle: kept sets and masks bit-exact, renormalised
values within 1e-6 absolute, valid flags exact."""
import numpy as np
import pytest

import workloads
from oracle import filters
from tests.helpers import GUARD_DEEP, ensure_built, guard_accept

pytestmark = pytest.mark.gpu
TOL = 1e-6


@pytest.fixture(scope="module")
def ms():
    ensure_built()
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import min_sampling_gb300
    return min_sampling_gb300


def _dev(x, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def _check_renorm(P, params, out, valid, fn):
    for i in range(P.shape[0]):
        exp, ok = fn(P[i], params[i])
        assert bool(valid[i]) == ok, (i, params[i])
        kept_gpu = out[i] != 0
        kept_ref = exp != 0
        assert np.array_equal(kept_gpu, kept_ref), (i, params[i], np.nonzero(kept_gpu ^ kept_ref)[0][:10])
        assert np.max(np.abs(out[i].astype(np.float64) - exp)) <= TOL, (i, params[i])


def _run(ms, kind, P, params, inplace=False, misalign=False):
    import torch
    x = _dev(P)
    if misalign:
        flat = torch.empty(P.size + 1, dtype=torch.float32, device="cuda")
        flat[1:] = x.reshape(-1)
        x = flat[1:].view(P.shape)
    dt = torch.float32 if kind == "top_p" else torch.int32
    p = _dev(np.asarray(params), dt)
    fn = {"top_k": ms.top_k_renorm_probs, "top_p": ms.top_p_renorm_probs, "mask": ms.top_k_mask_logits}[kind]
    out, valid = fn(x, p, out=x if inplace else None)
    torch.cuda.synchronize()
    return out.cpu().numpy(), valid.cpu().numpy()


def _softmax_rows(n, V, sigma, seed, accept=None):
    rows = []
    for i in range(n):
        for att in range(64):
            rng = workloads.row_rng(seed, i, att)
            p, _ = workloads.detie(workloads.softmax_fp32(rng.normal(0, sigma, V)))
            if accept is None or accept(i, p):
                break
        rows.append(p)
    return np.stack(rows)


def test_hand_rows(ms):
    P = np.array([[0.05, 0.40, 0.10, 0.30, 0.15]], np.float32)
    out, valid = _run(ms, "top_p", P, [0.8])
    assert np.allclose(out[0], [0, 0.40 / 0.85, 0, 0.30 / 0.85, 0.15 / 0.85], atol=TOL) and valid[0]
    out, valid = _run(ms, "top_k", P, [2])
    assert np.allclose(out[0], [0, 0.40 / 0.70, 0, 0.30 / 0.70, 0], atol=TOL) and valid[0]
    Q = np.array([[0.35, 0.28, 0.18, 0.12, 0.07]], np.float32)
    out, _ = _run(ms, "top_k", Q, [2])
    assert np.allclose(out[0], [0.35 / 0.63, 0.28 / 0.63, 0, 0, 0], atol=TOL)


def test_config1_rows_all_parameters(ms):
    w = workloads.config1()
    P = w.probs
    for k in [1, 2, 10, 50, 512, 1023, 1024, 0, -3, 5000]:
        out, valid = _run(ms, "top_k", P, [k] * 4)
        _check_renorm(P, [k] * 4, out, valid, filters.top_k_renorm)
    acc = guard_accept(lambda i: [(None, p, None, "joint") for p in (0.1, 0.5, 0.9, 0.95, 0.999)])
    P2 = _softmax_rows(4, 1024, 2.0, 555, acc)
    for p in [0.1, 0.5, 0.9, 0.95, 0.999, 1.0, 1.5, 0.0, -1.0]:
        out, valid = _run(ms, "top_p", P2, [p] * 4)
        _check_renorm(P2, [p] * 4, out, valid, filters.top_p_renorm)


@pytest.mark.parametrize("V", [1, 2, 3, 5, 127, 128, 511, 513, 1000, 4099, 70001])
def test_ragged_vocab_sizes(ms, V):
    rng = np.random.default_rng(V)
    ks = [int(x) for x in rng.integers(1, V + 1, 4)]
    ps = [float(x) for x in rng.uniform(0.05, 0.98, 4)]
    acc = guard_accept(lambda i: [(None, ps[i], None, "joint")])
    P = _softmax_rows(4, V, 2.5, 1000 + V, acc)
    out, valid = _run(ms, "top_k", P, ks)
    _check_renorm(P, ks, out, valid, filters.top_k_renorm)
    out, valid = _run(ms, "top_p", P, ps)
    _check_renorm(P, ps, out, valid, filters.top_p_renorm)
    Z = (rng.normal(0, 3, (4, V))).astype(np.float32)
    Z = np.stack([workloads.detie(z, positive_only=False)[0] for z in Z])
    out, valid = _run(ms, "mask", Z, ks)
    for i in range(4):
        exp, ok = filters.top_k_mask_logits(Z[i], ks[i])
        assert ok == bool(valid[i]) and np.array_equal(out[i], exp)


def test_misaligned_and_inplace(ms):
    P = _softmax_rows(3, 4096, 2.0, 77)
    out, valid = _run(ms, "top_k", P, [7, 70, 700], misalign=True)
    _check_renorm(P, [7, 70, 700], out, valid, filters.top_k_renorm)
    out, valid = _run(ms, "top_k", P, [7, 70, 700], inplace=True)
    _check_renorm(P, [7, 70, 700], out, valid, filters.top_k_renorm)
    acc = guard_accept(lambda i: [(None, 0.7, None, "joint")])
    P = _softmax_rows(3, 4096, 2.0, 78, acc)
    out, valid = _run(ms, "top_p", P, [0.7] * 3, inplace=True, misalign=True)
    _check_renorm(P, [0.7] * 3, out, valid, filters.top_p_renorm)


def test_invalid_rows(ms):
    P = _softmax_rows(5, 3000, 2.0, 91)
    P[1, 17] = np.nan
    P[2, 5] = -1e-3
    P[3, :] = 0
    for kind, fn, prm in [("top_k", filters.top_k_renorm, [10] * 5), ("top_p", filters.top_p_renorm, [0.9] * 5)]:
        out, valid = _run(ms, kind, P, prm)
        assert valid.tolist() == [1, 0, 0, 0, 1]
        assert not out[1:4].any()
    out, valid = _run(ms, "top_p", P, [0.9, 0.9, 0.9, 0.9, float("nan")])
    assert valid.tolist() == [1, 0, 0, 0, 0] and not out[4].any()
    Z = np.random.default_rng(3).normal(0, 2, (3, 999)).astype(np.float32)
    Z[1, 400] = np.nan
    out, valid = _run(ms, "mask", Z, [5, 5, 5])
    assert valid.tolist() == [1, 0, 1] and np.isneginf(out[1]).all()


def test_mask_special_values(ms):
    # Tie-free (+0 and -0 are equal values, so only one of them appears).
    z = np.array([0.0, -np.inf, np.inf, -1.5, 2.5, -3e38, 3e38, 1e-45, -1e-45], np.float32)
    Z = np.stack([z, z[::-1].copy()])
    for k in range(1, 9):
        out, valid = _run(ms, "mask", Z, [k, k])
        for i in range(2):
            exp, ok = filters.top_k_mask_logits(Z[i], k)
            assert np.array_equal(np.isneginf(out[i]), np.isneginf(exp)), (k, i)
            assert np.array_equal(out[i][~np.isneginf(exp)], exp[~np.isneginf(exp)])


def test_config3_full_size(ms):
    """B=64, V=151936, z ~ N(0, 3^2): top-k 50, top-p 0.9 and the logit mask."""
    # Plain top-p 0.9 cuts at a token of mass ~1.3e-5 here, so no row can keep both
    # neighbouring prefix masses 1e-5 from the target; that use gets the deep guard.
    acc = guard_accept(lambda i: [(None, 0.9, None, "joint", GUARD_DEEP), (50, 0.9, None, "top_k_first"),
                                  (50, 0.9, None, "joint")])
    w = workloads.config3(accept=acc)
    out, valid = _run(ms, "top_k", w.probs, [50] * 64)
    _check_renorm(w.probs, [50] * 64, out, valid, filters.top_k_renorm)
    assert (np.count_nonzero(out, axis=1) == 50).all()
    out, valid = _run(ms, "top_p", w.probs, [0.9] * 64)
    _check_renorm(w.probs, [0.9] * 64, out, valid, filters.top_p_renorm)
    out, valid = _run(ms, "mask", w.logits, [50] * 64)
    for i in range(64):
        exp, ok = filters.top_k_mask_logits(w.logits[i], 50)
        assert ok and valid[i] and np.array_equal(out[i], exp)


def test_large_k_bisection_path(ms):
    """k beyond the candidate capacity and beyond the segment count: the key bisection."""
    P = _softmax_rows(2, 200_000, 1.0, 123)
    for k in [3000, 60_000, 199_999]:
        out, valid = _run(ms, "top_k", P, [k, k])
        _check_renorm(P, [k, k], out, valid, filters.top_k_renorm)
    Z = np.stack([workloads.detie(np.random.default_rng(s).normal(0, 1, 200_000).astype(np.float32),
                                  positive_only=False)[0] for s in (1, 2)])
    for k in [3000, 150_000]:
        out, valid = _run(ms, "mask", Z, [k, k])
        for i in range(2):
            exp, ok = filters.top_k_mask_logits(Z[i], k)
            assert np.array_equal(out[i], exp)


def test_candidates_concentrated_in_one_cta(ms):
    """Most large values inside the first eighth of the row: the CTA that owns it has
    more top-k candidates than its share of the on-chip list, but the total fits, so
    every CTA collects again at exact offsets."""
    Z = workloads.concentrated_logits(2, 151936, 1000, 19000, seed=31)
    P = np.stack([workloads.detie(workloads.softmax_fp32(z))[0] for z in Z])
    for k in (100, 400):
        out, valid = _run(ms, "top_k", P, [k, k])
        _check_renorm(P, [k, k], out, valid, filters.top_k_renorm)
        out, valid = _run(ms, "mask", Z, [k, k])
        for i in range(2):
            exp, ok = filters.top_k_mask_logits(Z[i], k)
            assert np.array_equal(out[i], exp)


def test_max_vocab_row(ms):
    V = 2097152
    acc = guard_accept(lambda i: [(None, 0.5, None, "joint")])
    P = _softmax_rows(1, V, 2.0, 9, acc)
    out, valid = _run(ms, "top_k", P, [100])
    _check_renorm(P, [100], out, valid, filters.top_k_renorm)
    out, valid = _run(ms, "top_p", P, [0.5])
    _check_renorm(P, [0.5], out, valid, filters.top_p_renorm)


def _crowded_rows(V, seed):
    """Rows whose top values crowd into a few quarter-binade bins of the segment-maximum
    histogram, so that the coarse top-k bound admits more than 128 segments and is
    refined inside its bin: logits 12 + N(0, 1) (all in [8, 16) but the far tails),
    log-softmax logits of N(0, 3^2) (all negative), and near-flat probabilities
    softmax(N(0, 0.05^2)) (all within a few percent of 1/V)."""
    rng = np.random.default_rng([seed, V])
    z1 = workloads.detie((12.0 + rng.normal(0, 1, V)).astype(np.float32), positive_only=False)[0]
    z = rng.normal(0, 3, V)
    z2 = workloads.detie((z - (np.log(np.sum(np.exp(z - z.max()))) + z.max())).astype(np.float32),
                         positive_only=False)[0]
    p3 = workloads.detie(workloads.softmax_fp32(rng.normal(0, 0.05, V)))[0]
    return np.stack([z1, z2]), p3


@pytest.mark.parametrize("k", [1, 50, 300, 900])
def test_refined_bound_crowded_rows(ms, k):
    """The refined top-k bound (second histogram inside the boundary bin) and, for
    k = 300 and 900, candidate lists longer than the register path (the CTA's radix
    select): masks and renormalised rows against the oracle."""
    Z, p3 = _crowded_rows(151936, 5)
    out, valid = _run(ms, "mask", Z, [k, k])
    for i in range(2):
        exp, ok = filters.top_k_mask_logits(Z[i], k)
        assert ok and valid[i] and np.array_equal(out[i], exp), (k, i)
    P = np.stack([workloads.detie(workloads.softmax_fp32(Z[0]))[0], p3])
    out, valid = _run(ms, "top_k", P, [k, k])
    _check_renorm(P, [k, k], out, valid, filters.top_k_renorm)
    assert (np.count_nonzero(out, axis=1) == k).all()


def test_top_p_scales_and_extremes(ms):
    """Top-p renormalisation of rows scaled by exact powers of two (2^100, 2^-80:
    the integer mass scale follows the row maximum), of a row pushed into the
    subnormal range, and top_p from 0 (the maximum alone) to 0.95: kept sets
    bit-exact, values within 1e-6 of the oracle's."""
    ps = [0.0, 1e-4, 0.3, 0.5, 0.8, 0.95]
    acc = guard_accept(lambda i: [(None, p, None, "joint", GUARD_DEEP if p > 0.9 else 1e-5) for p in ps if p > 0])
    base = _softmax_rows(3, 50_000, 3.0, 77, acc)
    assert all(acc(i, base[i]) for i in range(3))
    for scale in (2.0 ** 100, 2.0 ** -80, 1.0):
        P = (base.astype(np.float64) * scale).astype(np.float32)
        assert np.array_equal(P.astype(np.float64) / scale, base.astype(np.float64))   # exact scaling
        for p in ps:
            out, valid = _run(ms, "top_p", P, [p] * 3)
            for i in range(3):
                exp, ok = filters.top_p_renorm(P[i], p)
                assert bool(valid[i]) == ok
                assert np.array_equal(out[i] != 0, exp != 0), (scale, p, i)
                assert np.max(np.abs(out[i].astype(np.float64) - exp)) <= TOL, (scale, p, i)
    # Subnormal values: the scaled row differs from `base` by rounding, so its own
    # boundary margins decide which top_p are checked.
    S = (base[:1].astype(np.float64) * 2.0 ** -135).astype(np.float32)
    M = float(S.astype(np.float64).sum())
    for p in (0.0, 0.3, 0.5, 0.8):
        if p > 0 and filters.topp_boundary_margin(S[0], None, p, None, "joint") < 1e-5 * M:
            continue
        out, valid = _run(ms, "top_p", S, [p])
        exp, ok = filters.top_p_renorm(S[0], p)
        assert ok and valid[0]
        assert np.array_equal(out[0] != 0, exp != 0), p
        assert np.max(np.abs(out[0].astype(np.float64) - exp)) <= TOL, p


def test_top_p_crowded_crossing_bin(ms):
    """Near-flat rows (softmax of N(0, 0.05^2), V = 20000): the bin of the top-p
    crossing holds thousands of elements, more than the leader's list, so every CTA
    finishes with the exact histogram passes.  Kept sets bit-exact, values within
    1e-6."""
    ps = [0.2, 0.5, 0.8]
    acc = guard_accept(lambda i: [(None, p, None, "joint") for p in ps])
    P = _softmax_rows(4, 20_000, 0.05, 91, acc)
    assert all(acc(i, P[i]) for i in range(4))
    keys = P.view(np.uint32) >> 21
    assert max(np.bincount(keys[i]).max() for i in range(4)) > 2048   # the crowded bin
    for p in ps:
        out, valid = _run(ms, "top_p", P, [p] * 4)
        _check_renorm(P, [p] * 4, out, valid, filters.top_p_renorm)
