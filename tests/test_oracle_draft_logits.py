"""Pins of the oracle's draft-logits mode ([spec-in-vllm] 7.1 probabilistic draft sampling with the
draft logits kept; 7.4 block stats over target and draft logits): q = softmax(draft_logits / T)
per draft row, then the same verification as with draft probabilities."""
import dataclasses

import numpy as np
import pytest
from scipy.special import softmax

import oracle
import workloads
from _util import binom_z, chi2_pvalue, draw_from, replicated_batch, to_bf16_bits

N = 200_000


def test_draft_probs_equal_a_float64_softmax():
    rng = np.random.default_rng(4)
    for V, dtype, T in [(7, "f32", 1.0), (1000, "f32", 0.6), (4099, "bf16", 1.4)]:
        K = [2, 0, 3]
        cu = np.concatenate([[0], np.cumsum(K)]).astype(np.int32)
        dl = (rng.standard_normal((int(cu[-1]), V)) * 3).astype(np.float32)
        raw = to_bf16_bits(dl) if dtype == "bf16" else dl
        exact = (raw.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else dl
        temp = np.full(3, T, np.float32)
        q = oracle.draft_probs(raw, dtype == "bf16", cu, temp, np.zeros(3, np.uint8))
        invT = np.float32(1.0) / np.float32(T)
        want = softmax((exact * invT).astype(np.float64), axis=1)
        np.testing.assert_allclose(q, want, rtol=3e-6, atol=1e-30)
        np.testing.assert_allclose(q.astype(np.float64).sum(1), 1.0, rtol=1e-5)
    # a greedy request's rows use T = 1 (never read, but defined)
    q = oracle.draft_probs(dl[:2], False, np.array([0, 2], np.int32), np.array([0.0], np.float32),
                           np.zeros(1, np.uint8))
    np.testing.assert_allclose(q, softmax(dl[:2].astype(np.float64), axis=1), rtol=3e-6)


def _logits_batch(V, K, T, seed, n=N):
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    dl = (logits[:K] + rng.standard_normal((K, V))).astype(np.float32)
    q = np.stack([softmax(dl[j].astype(np.float64) / T) for j in range(K)])
    d = np.stack([draw_from(q[j], n, seed=seed + 10 + j) for j in range(K)], axis=1)
    b = replicated_batch(logits, None, d, temperature=T, seed=seed + 99)
    b = dataclasses.replace(b, draft_logits=np.ascontiguousarray(np.tile(dl, (n, 1))))
    return b, logits, q


@pytest.mark.parametrize("V,T", [(4, 1.0), (8, 0.8), (16, 1.3)])
def test_lossless_with_draft_logits(V, T):
    K = 2
    b, logits, q = _logits_batch(V, K, T, seed=700 + V)
    o = oracle.run(b)
    p = [softmax(logits[j].astype(np.float64) / T) for j in range(K + 1)]
    s = o["sampled"]
    assert chi2_pvalue(np.bincount(s[:, 0], minlength=V), p[0]) > 1e-3
    sel = o["num_sampled"] >= 2
    assert chi2_pvalue(np.bincount(s[sel, 1], minlength=V), p[1]) > 1e-3
    # acceptance at position 0 happens with probability sum_v min(p_v, q_v)
    acc = o["num_sampled"] >= 2
    assert abs(binom_z(int(acc.sum()), N, float(np.minimum(p[0], q[0]).sum()))) < 4.5


def test_workload_style_batch_in_draft_logits_mode():
    b = workloads.make_batch(name="dl", data_seed=3, verify_seed=5, K=[3, 0, 5, 2], vocab_size=2000,
                             logits_dtype="bf16", sigma=2.5, zipf_coef=1.1, q_mode="logits",
                             q_noise=2.0, temperature=np.array([1.0, 0.7, 1.2, 0.0], np.float32))
    assert b.draft_probs is None and b.draft_logits.shape == (10, 2000)
    o = oracle.run(b)
    assert o["status"] == 0
    # a rejection inside a request emits a target-side token; greedy request 3 emits argmaxes
    assert np.all(o["num_sampled"] == o["jstar"] + 1)
    assert np.all((o["sampled"] >= -1) & (o["sampled"] < 2000))
