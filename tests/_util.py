"""Shared helpers of the test suite (fixtures parsing, batch construction, statistics)."""
from __future__ import annotations

import os

import numpy as np
from scipy import stats

from workloads import Batch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    """Parse a tests/golden/*.txt fixture: '#' comments, then 'key value...' lines."""
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            try:
                out[key] = [float(v) for v in vals]
            except ValueError:
                out[key] = vals
    return out


def replicated_batch(rows: np.ndarray, q_rows: np.ndarray | None, draft_ids: np.ndarray, *,
                     temperature: float = 1.0, greedy: bool = False, seed: int = 1234,
                     dtype: str = "f32") -> Batch:
    """N requests sharing the same K+1 logit rows (rows: [K+1, V]) and draft distributions
    (q_rows: [K, V] or None); draft_ids: [N, K]. RNG draws stay independent because they are
    keyed by the request index."""
    rows = np.asarray(rows, dtype=np.float32)
    K1, V = rows.shape
    K = K1 - 1
    draft_ids = np.asarray(draft_ids, dtype=np.int32).reshape(-1, K) if K else np.zeros((len(draft_ids), 0), np.int32)
    N = draft_ids.shape[0]
    logits = np.ascontiguousarray(np.tile(rows, (N, 1)))
    if dtype == "bf16":
        logits = to_bf16_bits(logits)
    q = None if q_rows is None else np.ascontiguousarray(np.tile(np.asarray(q_rows, np.float32), (N, 1)))
    cu = (np.arange(N + 1) * K).astype(np.int32)
    return Batch(name="replicated", logits=logits, logits_dtype=dtype, vocab_size=V,
                 draft_ids=draft_ids.reshape(-1).copy(), draft_probs=q, cu_num_draft=cu,
                 temperature=np.full(N, temperature, np.float32),
                 is_greedy=np.full(N, int(greedy), np.uint8), seed=seed)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def draw_from(p: np.ndarray, n: int, seed: int) -> np.ndarray:
    """n host-side draws from p (inverse CDF on numpy's generator): draft proposals."""
    rng = np.random.default_rng(seed)
    c = np.cumsum(np.asarray(p, np.float64))
    c /= c[-1]
    return np.minimum(np.searchsorted(c, rng.random(n), side="right"), len(p) - 1).astype(np.int32)


def chi2_pvalue(counts: np.ndarray, probs: np.ndarray) -> float:
    """Pearson chi-square goodness of fit; cells of zero probability must be empty."""
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    probs = probs / probs.sum()
    zero = probs == 0
    assert counts[zero].sum() == 0, f"mass on zero-probability cells: {counts[zero]}"
    exp = probs[~zero] * counts.sum()
    return float(stats.chisquare(counts[~zero], exp).pvalue)


def binom_z(successes: int, n: int, p: float) -> float:
    if p <= 0 or p >= 1:
        return 0.0 if (successes == 0 and p <= 0) or (successes == n and p >= 1) else float("inf")
    return (successes - n * p) / np.sqrt(n * p * (1 - p))
