"""Chain speculative-sampling verification, step by step.

TEST INFRASTRUCTURE ONLY.

The pages name speculative-decoding verification as a use of the sorting-free
sampler ([blog] section on community adoption) but give no algorithm, so this
module follows the published method:
  Y. Leviathan, M. Kalman, Y. Matias, "Fast Inference from Transformers via
  Speculative Decoding", ICML 2023: Algorithm 1 (one speculative step) and
  Appendix A.1 (the modified rejection sampling yields exactly the target
  distribution);
  C. Chen et al., "Accelerating Large Language Model Decoding with Speculative
  Sampling", 2023: Algorithm 2 (the same acceptance rule and residual).

One row: L draft tokens d_1..d_L (drawn by the caller from the draft rows
q_1..q_L) and L + 1 target rows p_1..p_{L+1}.
  for i = 1..L:
      accept d_i when u_i * q_i(d_i) < p_i(d_i)      (probability min(1, p/q));
      otherwise emit a token drawn from the residual max(p_i - q_i, 0) and stop;
  when all L are accepted, emit a token drawn from p_{L+1} (the bonus token).
The output holds the accepted draft tokens followed by the emitted token, L + 1
slots with -1 after the last one.

Readings (this library's; the pages are silent):
  - Rows are used as given (probabilities; nothing is renormalised).  The
    acceptance ratio and the residual are formed from the values as passed.
  - A draft token outside [0, V) is rejected.
  - Draws are the sampler's inverse transform over non-negative weights w: the
    first index j (index order) with w_j > 0 whose running sum exceeds u * sum(w)
    (dual_pivot.draw_inverse_transform with low = 0).
  - The uniforms come from the sampler's Philox stream of the row: round i
    (0-based) for the acceptance test of draft i, round L for the final draw.
  - When the weights of the final draw are not a valid row (a NaN or infinite
    value, a negative value in the bonus row, or no positive mass: a residual can
    only be empty when the draft and target rows disagree on their sums), no
    token is emitted and the slot holds -1.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

from .dual_pivot import draw_inverse_transform
from .filters import as64
from .philox import sampler_uniform


def residual_weights(p, q) -> np.ndarray:
    """max(p - q, 0) element by element (float64; exact for float32 inputs)."""
    return np.maximum(as64(p) - as64(q), 0.0)


def acceptance_probability(p, q) -> float:
    """Probability that a draft token drawn from q (normalised) is accepted:
    sum_x q(x) min(1, p(x) / q(x)) = sum_x min(p(x), q(x)) for normalised rows."""
    p64, q64 = as64(p), as64(q)
    qn = q64 / q64.sum()
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(qn > 0, np.minimum(1.0, p64 / np.where(qn > 0, qn, 1.0)), 0.0)
    return float(np.sum(qn * ratio))


def _draw(w: np.ndarray, u: float, bonus: bool) -> int:
    """The final draw over weights w, or -1 when w is not a valid row."""
    if not np.all(np.isfinite(w)) or (bonus and np.any(w < 0)):
        return -1
    total = float(np.sum(np.where(w > 0, w, 0.0)))
    if not (total > 0.0) or not math.isfinite(total):
        return -1
    return draw_inverse_transform(w, 0.0, u)


def verify(draft_probs, draft_tokens: Sequence[int], target_probs, u_accept: Sequence[float],
           u_final: float):
    """One row of chain verification.

    draft_probs: [L, V]; draft_tokens: [L]; target_probs: [L + 1, V];
    u_accept[i]: the uniform of draft i's acceptance test; u_final: the uniform of
    the final draw.  Returns (tokens [L + 1] with -1 padding, accepted count,
    emitted count).
    """
    q_rows = np.asarray(draft_probs, dtype=np.float32)
    p_rows = np.asarray(target_probs, dtype=np.float32)
    L = len(draft_tokens)
    V = p_rows.shape[1]
    out = np.full(L + 1, -1, np.int64)
    for i in range(L):
        d = int(draft_tokens[i])
        if 0 <= d < V:
            pd, qd = float(p_rows[i, d]), float(q_rows[i, d])
            # u has 24 bits and the rows are float32, so u * q is exact in float64.
            if float(u_accept[i]) * qd < pd:
                out[i] = d
                continue
        j = _draw(residual_weights(p_rows[i], q_rows[i]), u_final, bonus=False)
        out[i] = j
        return out, i, i + (1 if j >= 0 else 0)
    j = _draw(as64(p_rows[L]), u_final, bonus=True)
    out[L] = j
    return out, L, L + (1 if j >= 0 else 0)


def verify_philox(draft_probs, draft_tokens, target_probs, *, seed: int, offset: int, row: int):
    """``verify`` driven by the sampler's Philox stream of row ``row``: round i for
    the acceptance test of draft i, round L for the final draw."""
    L = len(draft_tokens)
    u_acc = [sampler_uniform(seed, offset, row, i) for i in range(L)]
    return verify(draft_probs, draft_tokens, target_probs, u_acc, sampler_uniform(seed, offset, row, L))


def first_emission_law(p, q) -> np.ndarray:
    """Exact law of the token emitted at the first position of a one-draft chain
    when the draft token is drawn from q (normalised) and the test and residual are
    those of ``verify``: for each draft token d, accept with probability
    min(1, p(d)/q(d)), else emit from the normalised residual.  (The theorem of
    Leviathan et al., Appendix A.1, says this equals p for normalised p and q.)"""
    p64, q64 = as64(p), as64(q)
    qn = q64 / q64.sum()
    r = residual_weights(p64, qn)
    rs = r.sum()
    rn = r / rs if rs > 0 else np.zeros_like(r)
    law = np.zeros_like(p64)
    for d in np.nonzero(qn > 0)[0]:
        a = min(1.0, p64[d] / qn[d])
        law[d] += qn[d] * a
        law += qn[d] * (1.0 - a) * rn
    return law


def accepted_count_law(draft_probs, target_probs) -> np.ndarray:
    """P(accepted = i), i = 0..L, when each draft token is drawn from its own
    (normalised) draft row and tested as in ``verify``, by enumerating every draft
    sequence (small V and L only): the chain stops at the first rejection."""
    q_rows = [as64(q) / as64(q).sum() for q in draft_probs]
    p_rows = [as64(p) for p in target_probs]
    L = len(q_rows)
    law = np.zeros(L + 1)

    def walk(i: int, prob: float):
        if i == L:
            law[L] += prob
            return
        for d in np.nonzero(q_rows[i] > 0)[0]:
            a = min(1.0, p_rows[i][d] / q_rows[i][d])
            walk(i + 1, prob * q_rows[i][d] * a)
            law[i] += prob * q_rows[i][d] * (1.0 - a)

    walk(0, 1.0)
    return law


def verify_rows(draft_probs, draft_tokens, target_probs, *, seed: int, offset: int,
                rows: Optional[Sequence[int]] = None):
    """``verify_philox`` over a batch: draft_probs [B, L, V], draft_tokens [B, L],
    target_probs [B, L + 1, V].  Returns (tokens [B, L + 1], accepted [B], emitted [B])."""
    B = np.asarray(draft_tokens).shape[0]
    L = np.asarray(draft_tokens).shape[1]
    idx = range(B) if rows is None else rows
    toks = np.full((len(idx), L + 1), -1, np.int64)
    acc = np.zeros(len(idx), np.int64)
    emi = np.zeros(len(idx), np.int64)
    for n, b in enumerate(idx):
        toks[n], acc[n], emi[n] = verify_philox(draft_probs[b], draft_tokens[b], target_probs[b],
                                                seed=seed, offset=offset, row=b)
    return toks, acc, emi
