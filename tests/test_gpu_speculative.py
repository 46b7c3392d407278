"""Parity of chain speculative-sampling verification (fs_chain_speculative_sampling)
with the oracle (oracle/speculative.py): the same Philox stream replayed row by row,
the law of the emitted token and of the accepted count over many chains, and the
edge cases."""
import numpy as np
import pytest

import workloads
from oracle import speculative as spec
from tests.helpers import chi2_pvalue, draws_for_tv, ensure_built, expected_null_tv, tv_distance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ms():
    ensure_built()
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import min_sampling_gb300
    return min_sampling_gb300


def _run(ms, draft, tokens, target, seed, offset):
    import torch
    d = torch.from_numpy(np.ascontiguousarray(draft)).cuda() if draft is not None else None
    t = torch.from_numpy(np.ascontiguousarray(tokens)).cuda() if tokens is not None else None
    p = torch.from_numpy(np.ascontiguousarray(target)).cuda()
    tok, acc, emi = ms.chain_speculative_sampling(d, t, p, seed=seed, offset=offset)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), acc.cpu().numpy(), emi.cpu().numpy()


def _agree(ms, draft, tokens, target, seed, offset, min_frac):
    tok, acc, emi = _run(ms, draft, tokens, target, seed, offset)
    rt, ra, re = spec.verify_rows(draft, tokens, target, seed=seed, offset=offset)
    same = (tok == rt).all(axis=1) & (acc == ra) & (emi == re)
    assert same.mean() >= min_frac, np.nonzero(~same)[0][:8]
    # every emitted token is one the method can emit: a draft token before the stop,
    # then a token of positive residual (or bonus) weight
    B, L = tokens.shape
    for b in range(B):
        a = int(acc[b])
        assert (tok[b, :a] == tokens[b, :a]).all() and (tok[b, a + 1:] == -1).all()
        j = int(tok[b, a])
        assert j >= 0 and emi[b] == a + 1
        w = (spec.residual_weights(target[b, a], draft[b, a]) if a < L
             else target[b, L].astype(np.float64))
        assert w[j] > 0
    return tok, acc


@pytest.mark.parametrize("L", [1, 4])
def test_full_size_replay(ms, L):
    """B = 64 rows of the Qwen vocabulary (V = 151936): the kernel and the oracle,
    driven by the same Philox stream, emit the same tokens."""
    draft, tokens, target = workloads.speculative_batch(64, L, 151936, seed=5)
    tok, acc = _agree(ms, draft, tokens, target, seed=2024, offset=7, min_frac=63 / 64)
    assert 0 < acc.mean() < L   # both accepted and rejected drafts occur


def test_ragged_vocab_and_scalar_path(ms):
    """V = 40001 (not a multiple of 4: the scalar path) and a small vocabulary."""
    for V in (40001, 130):
        draft, tokens, target = workloads.speculative_batch(16, 3, V, seed=V)
        _agree(ms, draft, tokens, target, seed=9, offset=V, min_frac=15 / 16)


def test_law_over_many_chains(ms):
    """One (draft, target) pair replicated over 10^6+ chains, draft tokens drawn from
    q per chain: the first emitted token follows p_1 (TV <= 0.005, chi-square), the
    accepted count follows the enumerated law (chi-square)."""
    import torch
    L, V = 2, 32
    draft1, _, target1 = workloads.speculative_batch(1, L, V, seed=3, sigma=1.0, drift=1.0)
    p1 = target1[0, 0].astype(np.float64)
    n = draws_for_tv(p1 / p1.sum())
    rng = np.random.default_rng(99)
    qn = draft1[0].astype(np.float64) / draft1[0].astype(np.float64).sum(axis=1, keepdims=True)
    tokens = np.stack([rng.choice(V, size=n, p=qn[i]) for i in range(L)], axis=1).astype(np.int32)
    d = torch.from_numpy(draft1).cuda().expand(n, L, V).contiguous()
    p = torch.from_numpy(target1).cuda().expand(n, L + 1, V).contiguous()
    tok, acc, emi = ms.chain_speculative_sampling(d, torch.from_numpy(tokens).cuda(), p, seed=77, offset=1)
    tok, acc, emi = tok.cpu().numpy(), acc.cpu().numpy(), emi.cpu().numpy()
    del d, p
    assert (emi == acc + 1).all() and (tok[np.arange(n), acc] >= 0).all()
    counts = np.bincount(tok[:, 0], minlength=V).astype(np.float64)
    law = spec.first_emission_law(target1[0, 0], draft1[0, 0])
    tv = tv_distance(counts, law)
    assert tv <= 0.005, (tv, expected_null_tv(law, n))
    assert chi2_pvalue(counts, law) > 1e-3
    acc_law = spec.accepted_count_law(draft1[0], target1[0])
    assert chi2_pvalue(np.bincount(acc, minlength=L + 1).astype(np.float64), acc_law) > 1e-3


def test_edge_cases(ms):
    rng = np.random.default_rng(4)
    V = 1000
    draft, tokens, target = workloads.speculative_batch(6, 3, V, seed=11)
    # row 0: q = p at every position, so every draft is accepted
    target[0, :3] = draft[0]
    # row 1: p(d) = 0 at the first position: rejected whatever u is
    target[1, 0, tokens[1, 0]] = 0.0
    # row 2: an out-of-range draft token at position 1
    tokens[2, 1] = V + 5
    # row 3: residual with no mass at position 0 (target equals draft there, token out
    # of range so the position is rejected): nothing is emitted
    target[3, 0] = draft[3, 0]
    tokens[3, 0] = -1
    # row 4: a NaN in the residual row of position 0 (draft token forced out of range)
    tokens[4, 0] = V
    target[4, 0, 17] = np.nan
    tok, acc, emi = _run(ms, draft, tokens, target, seed=5, offset=0)
    rt, ra, re = spec.verify_rows(draft, tokens, target, seed=5, offset=0)
    assert acc[0] == 3 and emi[0] == 4 and (tok[0, :3] == tokens[0]).all()
    assert acc[1] == 0 and tok[1, 0] != tokens[1, 0] and emi[1] == 1
    assert acc[2] <= 1
    assert acc[3] == 0 and emi[3] == 0 and (tok[3] == -1).all()
    assert acc[4] == 0 and emi[4] == 0 and (tok[4] == -1).all()
    assert (tok == rt).all() and (acc == ra).all() and (emi == re).all()
    # num_draft = 0: one draw from the single target row, as the oracle's
    t0 = target[:, :1].copy()
    tok, acc, emi = _run(ms, None, None, t0, seed=8, offset=3)
    rt, ra, re = spec.verify_rows(np.zeros((6, 0, V), np.float32), np.zeros((6, 0), np.int32), t0, seed=8, offset=3)
    assert (tok == rt).all() and (acc == 0).all() and (emi == re).all()
    assert emi[4] == 0 and (emi[[0, 1, 2, 3, 5]] == 1).all()   # row 4 still holds its NaN
    # empty batch
    import torch
    out = ms.chain_speculative_sampling(torch.zeros((0, 2, V), device="cuda"), torch.zeros((0, 2), dtype=torch.int32,
                                        device="cuda"), torch.zeros((0, 3, V), device="cuda"), seed=1, offset=0)
    assert out[0].shape == (0, 3)


def test_determinism_and_offsets(ms):
    draft, tokens, target = workloads.speculative_batch(32, 4, 5000, seed=21)
    a = _run(ms, draft, tokens, target, seed=1, offset=10)
    b = _run(ms, draft, tokens, target, seed=1, offset=10)
    c = _run(ms, draft, tokens, target, seed=1, offset=11)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[0], c[0])
