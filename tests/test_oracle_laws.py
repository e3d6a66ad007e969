"""Distributional pins of the oracle: losslessness (the output law equals p), the
accepted-length law, greedy and Gumbel-max special cases, and the target-side rule."""
import numpy as np
import pytest

import oracle
from _util import binom_z, chi2_pvalue, draw_from, replicated_batch

N = 200_000


def _softmax(x, T=1.0):
    z = np.asarray(x, np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def _rows(V, K, seed, sigma=1.5):
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((K + 1, V)) * sigma).astype(np.float32)
    qz = logits[:K].astype(np.float64) + rng.standard_normal((K, V))
    q = np.stack([_softmax(z) for z in qz]).astype(np.float32)
    return logits, q


@pytest.mark.parametrize("V,T", [(3, 1.0), (4, 0.7), (5, 1.3), (8, 1.0), (16, 0.9)])
def test_lossless_with_draft_probs(V, T):
    K = 2
    logits, q = _rows(V, K, seed=100 + V)
    d = np.stack([draw_from(q[j], N, seed=200 + 10 * V + j) for j in range(K)], axis=1)
    b = replicated_batch(logits, q, d, temperature=T, seed=400 + V)
    o = oracle.run(b)
    p = [_softmax(logits[j], T) for j in range(K + 1)]
    s = o["sampled"]
    assert chi2_pvalue(np.bincount(s[:, 0], minlength=V), p[0]) > 1e-3
    sel = o["num_sampled"] >= 2                # position 0 accepted: next output ~ p_1
    assert chi2_pvalue(np.bincount(s[sel, 1], minlength=V), p[1]) > 1e-3
    sel = o["num_sampled"] == 3                # both accepted: the bonus ~ p_2
    assert chi2_pvalue(np.bincount(s[sel, 2], minlength=V), p[2]) > 1e-3


@pytest.mark.parametrize("V", [3, 8, 16])
def test_lossless_without_draft_probs(V):
    K = 2
    logits, _ = _rows(V, K, seed=300 + V)
    rng = np.random.default_rng(V)
    d = rng.integers(0, V, size=(N, K)).astype(np.int32)   # any proposal rule
    b = replicated_batch(logits, None, d, temperature=1.0, seed=500 + V)
    o = oracle.run(b)
    s = o["sampled"]
    assert chi2_pvalue(np.bincount(s[:, 0], minlength=V), _softmax(logits[0])) > 1e-3
    # joint law of (accepted, token) equals "t ~ p; accept iff t == d" at position 0
    acc = o["num_sampled"] >= 2
    assert np.all(s[acc, 0] == d[acc, 0]) and np.all(s[~acc, 0] != d[~acc, 0])
    p0 = _softmax(logits[0])
    assert abs(binom_z(acc.sum(), N, float(np.mean(p0[d[:, 0]])))) < 4.5


def test_gumbel_max_non_speculative():
    for V, T in [(5, 1.0), (16, 0.5), (16, 2.0)]:
        rng = np.random.default_rng(V)
        row = (rng.standard_normal((1, V)) * 2).astype(np.float32)
        b = replicated_batch(row, None, np.zeros((N, 0), np.int32), temperature=T, seed=600 + V)
        o = oracle.run(b)
        assert np.all(o["num_sampled"] == 1) and np.all(o["num_rejected"] == 0)
        assert chi2_pvalue(np.bincount(o["sampled"][:, 0], minlength=V), _softmax(row[0], T)) > 1e-3


def test_greedy_outputs_are_argmax():
    V, K = 16, 3
    logits, q = _rows(V, K, seed=7)
    logits[1, 4] = logits[1, 11] = logits[1].max() + 1     # tie: the lower index is the argmax
    amax = [int(np.argmax(r)) for r in logits]
    rng = np.random.default_rng(8)
    d = np.where(rng.random((2000, K)) < 0.6, np.array(amax[:K]), rng.integers(0, V, (2000, K)))
    b = replicated_batch(logits, q, d.astype(np.int32), greedy=True, seed=9)
    o = oracle.run(b)
    for i in range(2000):
        n = o["num_sampled"][i]
        for j in range(n):
            assert o["sampled"][i, j] == amax[j]
        exp_n = next((j + 1 for j in range(K) if d[i, j] != amax[j]), K + 1)
        assert n == exp_n


def test_accepted_length_law():
    V, K = 8, 3
    logits, q = _rows(V, K, seed=21)
    p = [_softmax(logits[j]) for j in range(K)]
    d = np.array([int(np.argmax(q[j] / p[j])) for j in range(K)])   # tokens the draft over-weights
    a = [min(1.0, p[j][d[j]] / q[j][d[j]]) for j in range(K)]
    b = replicated_batch(logits, q, np.tile(d, (N, 1)), seed=22)
    o = oracle.run(b)
    length = o["num_sampled"] - 1
    for k in range(1, K + 1):
        assert abs(binom_z(int((length >= k).sum()), N, float(np.prod(a[:k])))) < 4.5
    assert np.all((o["num_sampled"] == K + 1) == (o["num_rejected"] == 0))
    assert np.all(o["num_rejected"] == K - length)


def test_rejection_emits_target_side_token():
    """With draft probs the token at a rejection has positive residual weight; the rejected
    draft token itself can only come back if p > q there."""
    V, K = 32, 2
    logits, q = _rows(V, K, seed=41)
    d = np.stack([draw_from(q[j], 20_000, seed=50 + j) for j in range(K)], axis=1)
    b = replicated_batch(logits, q, d, seed=42)
    o = oracle.run(b)
    rr = [oracle.residual_row(logits[j], False, 1.0, q[j])[1] for j in range(K)]
    rej = o["num_rejected"] > 0
    j = o["jstar"][rej]
    tok = o["sampled"][rej, :][np.arange(rej.sum()), j]
    assert np.all(np.array([rr[jj][t] for jj, t in zip(j, tok)]) > 0)
