"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark.

This module only makes data.  It holds none of the sampling method's arithmetic:
no allowed sets, thresholds, prefix masses or draws.  Both the CPU oracle and the
CUDA library are fed from here and neither is imported by it.

Every generator is deterministic in its seed.  Row ``i`` of a matrix is drawn from
``numpy.random.default_rng([seed, i, attempt])`` so that one row can be redrawn
(``attempt`` + 1) without disturbing the others; callers that must reject a row
(for example the tests' top-p boundary guard, which needs the oracle) pass an
``accept(row_index, row) -> bool`` callback.

Workload shapes follow the pages' workloads (the Qwen vocabulary of 151936 on the
F4 drill page, the 32K/128K vocabularies and the "sharp / flat / long-tail"
distribution shapes listed in the performance-testing section of the sorting-free
sampling explainer).  No public dataset is involved; these arrays stand in for
model outputs.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Optional

import numpy as np

SEED_BASE = 20261202


def cfg_seed(cfg_id: int, block: int = 0) -> int:
    """Seed of configuration ``cfg_id`` (1-based), row block ``block``."""
    return SEED_BASE + 1000 * cfg_id + block


def row_rng(seed: int, row: int, attempt: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed) & 0xFFFFFFFF, int(row), int(attempt)])


def softmax_fp32(z: np.ndarray) -> np.ndarray:
    """exp(z - max) / sum, evaluated in float64 and rounded once to float32."""
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(z - z.max())
    return (e / e.sum()).astype(np.float32)


def _order_key(x: np.ndarray) -> np.ndarray:
    """Monotone map of float32 values to int64 keys (sign-aware bit pattern)."""
    u = x.view(np.uint32).astype(np.int64)
    neg = u >= 0x80000000
    return np.where(neg, 0xFFFFFFFF - u, u + 0x80000000)


def _from_order_key(k: np.ndarray) -> np.ndarray:
    u = np.where(k >= 0x80000000, k - 0x80000000, 0xFFFFFFFF - k).astype(np.uint32)
    return u.view(np.float32)


def detie(x: np.ndarray, positive_only: bool = True) -> tuple[np.ndarray, int]:
    """Make the float32 values of ``x`` pairwise distinct.

    Values are visited in ascending order and each one is raised, if needed, to the
    next representable float32 above its (already raised) predecessor:
    key'[i] = max(key[i], key'[i-1] + 1), computed in closed form as
    i + running-max(key[j] - j).  With ``positive_only`` zeros and negatives are left
    alone (they are never sampled).  Returns the new array and the number of raised
    entries.
    """
    x = np.array(x, dtype=np.float32, copy=True)
    order = np.argsort(x, kind="stable")
    s = x[order]
    start = int(np.searchsorted(s, np.float32(0.0), side="right")) if positive_only else 0
    body = s[start:]
    if body.size < 2:
        return x, 0
    key = _order_key(body)
    idx = np.arange(key.size, dtype=np.int64)
    new = np.maximum.accumulate(key - idx) + idx
    bumps = int(np.count_nonzero(new != key))
    if bumps:
        s[start:] = _from_order_key(new)
        x[order] = s
    return x, bumps


def has_positive_ties(x: np.ndarray) -> bool:
    v = np.asarray(x, dtype=np.float32)
    v = v[v > 0]
    return np.unique(v).size != v.size


@dataclasses.dataclass
class Workload:
    """One batch of synthetic input plus the per-output-row parameters."""

    name: str
    probs: np.ndarray                      # [B_in, V] float32
    top_k: np.ndarray                      # [B_out] int32 (<= 0 or >= V: no top-k)
    top_p: np.ndarray                      # [B_out] float32 (>= 1: no top-p)
    min_p: np.ndarray                      # [B_out] float32 (<= 0: no min-p)
    indices: Optional[np.ndarray] = None   # [B_out] int32 output row -> input row
    logits: Optional[np.ndarray] = None    # [B_in, V] float32 (mask_logits input)
    bad_rows: Optional[np.ndarray] = None  # input rows made all-zero or NaN
    order: str = "joint"
    bumps: int = 0
    meta: dict = dataclasses.field(default_factory=dict)

    @property
    def batch_in(self) -> int:
        return int(self.probs.shape[0])

    @property
    def batch_out(self) -> int:
        return int(self.top_k.shape[0])

    @property
    def vocab(self) -> int:
        return int(self.probs.shape[1])


Accept = Optional[Callable[[int, np.ndarray], bool]]


def _rows(n: int, seed: int, draw: Callable[[np.random.Generator, int], np.ndarray],
          accept: Accept, max_attempts: int = 64) -> tuple[list[np.ndarray], int, int]:
    rows, bumps, redraws = [], 0, 0
    for i in range(n):
        for attempt in range(max_attempts):
            row = draw(row_rng(seed, i, attempt), i)
            if accept is None or accept(i, row):
                break
            redraws += 1
        else:
            raise RuntimeError(f"row {i}: no acceptable draw in {max_attempts} attempts")
        rows.append(row)
    return rows, bumps, redraws


# ---------------------------------------------------------------------------
# The pages' hand rows (worked examples).
# ---------------------------------------------------------------------------

HAND_ROWS = {
    # F4 drill page, section 1: top-p 0.8 keeps 0.40, 0.30, 0.15.
    "f4_topp": np.array([0.05, 0.40, 0.10, 0.30, 0.15], dtype=np.float32),
    # Explainer, "a simplified top-k example": top-k 2 keeps A and B.
    "explainer_topk": np.array([0.35, 0.28, 0.18, 0.12, 0.07], dtype=np.float32),
    # Explainer, "filter order changes the distribution": top-k 3, top-p 0.6.
    "explainer_order": np.array([0.40, 0.30, 0.20, 0.10], dtype=np.float32),
}


# ---------------------------------------------------------------------------
# Configurations.
# ---------------------------------------------------------------------------

def config1(seed: Optional[int] = None, accept: Accept = None) -> Workload:
    """B=4, V=1024, z ~ N(0, 2^2), p = softmax(z); rows with a duplicate value are redrawn.

    Per-row (top_k, top_p, min_p) = (1, 1.0, 0), (10, 0.9, 0), (50, 0.95, 0.1), (1024, 0.5, 0).
    """
    seed = cfg_seed(1) if seed is None else seed
    V = 1024

    def draw(rng, i):
        while True:
            p = softmax_fp32(rng.normal(0.0, 2.0, V))
            if not has_positive_ties(p):
                return p

    rows, _, redraws = _rows(4, seed, draw, accept)
    probs = np.stack(rows)
    zs = np.stack([row_rng(seed + 7, i).normal(0.0, 2.0, V) for i in range(4)]).astype(np.float32)
    logits = np.stack([detie(z, positive_only=False)[0] for z in zs])
    return Workload(
        name="c1_b4_v1024", probs=probs,
        top_k=np.array([1, 10, 50, 1024], dtype=np.int32),
        top_p=np.array([1.0, 0.9, 0.95, 0.5], dtype=np.float32),
        min_p=np.array([0.0, 0.0, 0.1, 0.0], dtype=np.float32),
        logits=logits, meta={"redraws": redraws})


def config2(seed: Optional[int] = None, accept: Accept = None, batch: int = 64,
            vocab: int = 32000) -> Workload:
    """B=64, V=32000, p = softmax(z / T_b), z ~ N(0,1), T_b ~ U[0.3, 1.5].

    Joint top-k + top-p with top_k ~ U{1..100}, top_p ~ U[0.7, 1.0] per row.
    """
    seed = cfg_seed(2) if seed is None else seed
    prng = np.random.default_rng([seed, 999_999])
    temps = prng.uniform(0.3, 1.5, batch)
    top_k = prng.integers(1, 101, batch).astype(np.int32)
    top_p = prng.uniform(0.7, 1.0, batch).astype(np.float32)
    bumps = [0]

    def draw(rng, i):
        p, nb = detie(softmax_fp32(rng.normal(0.0, 1.0, vocab) / temps[i]))
        bumps[0] += nb
        return p

    rows, _, redraws = _rows(batch, seed, draw, accept)
    return Workload(
        name=f"c2_b{batch}_v{vocab}", probs=np.stack(rows), top_k=top_k, top_p=top_p,
        min_p=np.zeros(batch, np.float32), order="joint", bumps=bumps[0],
        meta={"redraws": redraws, "temps": temps})


def config3(seed: Optional[int] = None, accept: Accept = None, batch: int = 64,
            vocab: int = 151936, with_logits: bool = True) -> Workload:
    """B=64, V=151936 (the Qwen vocabulary), z ~ N(0, 3^2), p = softmax(z).

    top_k = 50, top_p = 0.9 on every row; the same matrix feeds the top-k-first
    sampler, both renormalisers and (through ``logits`` = z) the logit mask.
    """
    seed = cfg_seed(3) if seed is None else seed
    zs = {}
    bumps = [0]

    def draw(rng, i):
        z = rng.normal(0.0, 3.0, vocab)
        zs[i] = z
        p, nb = detie(softmax_fp32(z))
        bumps[0] += nb
        return p

    rows, _, redraws = _rows(batch, seed, draw, accept)
    logits = None
    if with_logits:
        logits = np.stack([detie(zs[i].astype(np.float32), positive_only=False)[0]
                           for i in range(batch)])
    return Workload(
        name=f"c3_b{batch}_v{vocab}", probs=np.stack(rows),
        top_k=np.full(batch, 50, np.int32), top_p=np.full(batch, 0.9, np.float32),
        min_p=np.zeros(batch, np.float32), logits=logits, order="top_k_first",
        bumps=bumps[0], meta={"redraws": redraws})


def config4(batch_in: int = 1, seed: Optional[int] = None, accept: Accept = None,
            vocab: int = 128256, samples_per_row: int = 4) -> Workload:
    """V=128256, z = 2 * Student-t(3), p = softmax(z); fp32 underflow zeros are kept.

    ``indices`` maps ``samples_per_row`` output rows to each input row (parallel
    samples).  Parameters: min_p = 0.05 and top_p = 0.95 (the two entries are run
    separately; both arrays are filled).
    """
    seed = cfg_seed(4, batch_in) if seed is None else seed
    bumps = [0]

    def draw(rng, i):
        p, nb = detie(softmax_fp32(2.0 * rng.standard_t(3, vocab)))
        bumps[0] += nb
        return p

    rows, _, redraws = _rows(batch_in, seed, draw, accept)
    b_out = batch_in * samples_per_row
    return Workload(
        name=f"c4_b{batch_in}_v{vocab}", probs=np.stack(rows),
        top_k=np.zeros(b_out, np.int32), top_p=np.full(b_out, 0.95, np.float32),
        min_p=np.full(b_out, 0.05, np.float32),
        indices=np.repeat(np.arange(batch_in, dtype=np.int32), samples_per_row),
        bumps=bumps[0], meta={"redraws": redraws})


def config5(seed: Optional[int] = None, accept: Accept = None, batch: int = 256,
            vocab: int = 256000, bad_fraction: float = 0.05) -> Workload:
    """B=256, V=256000 adversarial mix.

    Rows [0, B/2): Zipf(s=1.1) over ranks 1..V, normalised and randomly permuted.
    Rows [B/2, B): near-flat softmax(z), z ~ N(0, 0.1^2).
    A seeded 5% of the rows is made all-zero or gets one NaN.
    Joint filters: top_k = V/2, top_p = 0.99, min_p = 0.01.
    """
    seed = cfg_seed(5) if seed is None else seed
    half = batch // 2
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    zipf = ranks ** -1.1
    zipf /= zipf.sum()
    bumps = [0]

    def draw(rng, i):
        if i < half:
            p = zipf[rng.permutation(vocab)].astype(np.float32)
        else:
            p = softmax_fp32(rng.normal(0.0, 0.1, vocab))
        p, nb = detie(p)
        bumps[0] += nb
        return p

    rows, _, redraws = _rows(batch, seed, draw, accept)
    probs = np.stack(rows)
    brng = np.random.default_rng([seed, 424242])
    n_bad = int(round(bad_fraction * batch))
    bad = np.sort(brng.choice(batch, n_bad, replace=False)).astype(np.int32)
    for r in bad:
        if brng.random() < 0.5:
            probs[r, :] = 0.0
        else:
            probs[r, int(brng.integers(0, vocab))] = np.float32(np.nan)
    return Workload(
        name=f"c5_b{batch}_v{vocab}", probs=probs,
        top_k=np.full(batch, vocab // 2, np.int32), top_p=np.full(batch, 0.99, np.float32),
        min_p=np.full(batch, 0.01, np.float32), bad_rows=bad, order="joint",
        bumps=bumps[0], meta={"redraws": redraws})


def random_small_rows(n: int, vocab: int, seed: int, zero_prob: float = 0.0) -> np.ndarray:
    """``n`` tie-free rows of ``vocab`` positive-or-zero float32 values (unnormalised
    scores drawn log-uniformly over two decades, optionally with exact zeros)."""
    rng = np.random.default_rng([seed, n, vocab])
    out = np.empty((n, vocab), np.float32)
    for i in range(n):
        while True:
            row = (10.0 ** rng.uniform(-2.0, 0.0, vocab)).astype(np.float32)
            if zero_prob > 0:
                row[rng.random(vocab) < zero_prob] = 0.0
            if not has_positive_ties(row):
                break
        out[i] = row
    return out


def concentrated_logits(n: int, vocab: int, n_big: int, span: int, seed: int, shift: float = 8.0) -> np.ndarray:
    """``n`` tie-free logit rows, z ~ N(0, 1), in which ``n_big`` entries at distinct
    random positions inside ``[0, span)`` are raised by ``shift``: most of a row's
    large values then sit in one part of it (a stress case for work split by index
    ranges)."""
    out = np.empty((n, vocab), np.float32)
    for i in range(n):
        rng = row_rng(seed, i)
        z = rng.normal(0.0, 1.0, vocab)
        z[rng.choice(span, size=n_big, replace=False)] += shift
        out[i] = detie(z.astype(np.float32), positive_only=False)[0]
    return out


def speculative_batch(batch: int, num_draft: int, vocab: int, seed: int, sigma: float = 3.0,
                      drift: float = 1.0):
    """Synthetic chain-verification inputs: target rows p = softmax(z), draft rows
    q = softmax(z + drift * N(0, 1)) (a draft model close to the target), and draft
    tokens drawn from q.  Returns (draft [B, L, V], tokens [B, L] int32, target
    [B, L + 1, V]), all float32 rows de-tied like the other workloads."""
    rng = np.random.default_rng([seed, batch, num_draft, vocab])
    target = np.empty((batch, num_draft + 1, vocab), np.float32)
    draft = np.empty((batch, num_draft, vocab), np.float32)
    tokens = np.empty((batch, num_draft), np.int32)
    for b in range(batch):
        for i in range(num_draft + 1):
            z = rng.normal(0.0, sigma, vocab)
            target[b, i] = detie(softmax_fp32(z))[0]
            if i < num_draft:
                q = detie(softmax_fp32(z + drift * rng.normal(0.0, 1.0, vocab)))[0]
                draft[b, i] = q
                q64 = q.astype(np.float64)
                tokens[b, i] = rng.choice(vocab, p=q64 / q64.sum())
    return draft, tokens, target
