"""Pins of the oracle's binary32 exp/log (the functions inside every decision) and of its
softmax statistics, against float64 library results."""
import numpy as np

import oracle
from _util import bf16_bits_to_f32, to_bf16_bits


def _ulps(got, exact):
    exact = np.asarray(exact, np.float64)
    ulp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    return np.abs(np.asarray(got, np.float64) - exact) / ulp


def test_exp_within_one_ulp():
    x = np.concatenate([
        np.linspace(-87.0, 0.0, 1_000_001, dtype=np.float32),
        -np.abs(np.random.default_rng(0).standard_normal(300_000)).astype(np.float32) * 10,
        np.linspace(0.0, 88.0, 10_001, dtype=np.float32),
        np.float32([0.0, -0.0, -1e-30, -1e-7, -87.0]),
    ])
    e = oracle.exp32_n(x)
    assert _ulps(e, np.exp(x.astype(np.float64))).max() <= 1.0
    assert oracle.exp32(0.0) == 1.0
    assert oracle.exp32(-87.01) == 0.0 and oracle.exp32(-1e30) == 0.0  # defined as 0 below -87
    assert oracle.exp32(89.0) == float("inf")


def test_log_within_two_ulp():
    rng = np.random.default_rng(1)
    bits = rng.integers(1, 0x7F800000, 1_000_000, dtype=np.uint64).astype(np.uint32)
    x = np.concatenate([bits.view(np.float32),                       # includes subnormals
                        np.linspace(0.5, 2.0, 500_001, dtype=np.float32),
                        np.float32([1.0, 1 - 2**-24, 1 + 2**-23, 2**-24, 16.6355, 2**-149])])
    lg = oracle.log32_n(x)
    assert _ulps(lg, np.log(x.astype(np.float64))).max() <= 2.0
    assert oracle.log32(1.0) == 0.0
    assert oracle.log32(1 - 2**-24) < 0.0                            # no collapse near 1
    assert oracle.log32(0.0) == float("-inf")
    assert np.isnan(oracle.log32(-1.0))


def _brute_stats(row_f32, invT):
    x = (row_f32 * np.float32(invT)).astype(np.float32)
    m = x.max()
    S = np.sum(np.exp(x.astype(np.float64) - np.float64(m)))
    return m, S, int(np.argmax(row_f32))


def test_row_stats_against_brute_force():
    rng = np.random.default_rng(5)
    for V, T, dtype in [(7, 1.0, "f32"), (64, 0.37, "f32"), (1000, 1.7, "bf16"), (1024, 0.8, "bf16"),
                        (333, 1.0, "bf16")]:
        n = 6
        rows = (rng.standard_normal((n, V)) * 3).astype(np.float32)
        rows[0, 5 % V] = rows[0].max() + 1.0   # unique max
        if V > 10:
            rows[1, 3] = rows[1, 9] = rows[1].max() + 2.0   # tie: lowest index wins
        logits = to_bf16_bits(rows) if dtype == "bf16" else rows
        vals = bf16_bits_to_f32(logits) if dtype == "bf16" else rows
        from _util import replicated_batch  # noqa
        from workloads import Batch
        b = Batch(name="t", logits=logits, logits_dtype=dtype, vocab_size=V,
                  draft_ids=np.zeros(n - 1, np.int32), draft_probs=None,
                  cu_num_draft=np.array([0, n - 1], np.int32), temperature=np.float32([T]),
                  is_greedy=np.uint8([0]), seed=1)
        o = oracle.run(b)
        invT = np.float32(1.0) / np.float32(T)
        for r in range(n):
            m, S, amax = _brute_stats(vals[r], invT)
            assert o["row_max"][r] == m                              # exact
            assert abs(o["row_sumexp"][r] - S) <= 1e-6 * S          # relative
            assert o["row_argmax"][r] == amax                        # lowest index on ties
        if V > 10:
            assert o["row_argmax"][1] == 3


def test_probabilities_sum_to_one_and_residual_identity():
    """p_v = t_v / S sums to 1; the race's residual weights rr_v / S equal max(0, p_v - q_v)
    where positive, and min(q, p) + max(0, p - q) = p, sum max(0, p - q) = 1 - sum min(p, q)."""
    rng = np.random.default_rng(11)
    for V in (3, 16, 1000, 32000):
        logits = (rng.standard_normal(V) * 2.5).astype(np.float32)
        z = logits.astype(np.float64) + rng.standard_normal(V)
        q = np.exp(z - z.max())
        q = (q / q.sum()).astype(np.float32)
        for T in (1.0, 0.6):
            invT = np.float32(1) / np.float32(T)
            t, rr, m, S = oracle.residual_row(logits, False, invT, q)
            p = t.astype(np.float64) / np.float64(S)
            assert abs(p.sum() - 1.0) < 1e-6
            x = (logits * invT).astype(np.float64)
            p_exact = np.exp(x - x.max()) / np.exp(x - x.max()).sum()
            assert np.max(np.abs(p - p_exact)) < 1e-6
            r = rr.astype(np.float64) / np.float64(S)
            qd = q.astype(np.float64)
            assert np.max(np.abs(np.maximum(r, 0) - np.maximum(p - qd, 0))) < 1e-6
            assert np.max(np.abs(np.minimum(qd, p) + np.maximum(r, 0) - p)) < 1e-6
            assert abs(np.maximum(r, 0).sum() - (1 - np.minimum(p, qd).sum())) < 1e-6
            clear = np.abs(p - qd) > 1e-6                             # sign of rr follows p - q
            assert np.all((rr[clear] > 0) == (p[clear] > qd[clear]))
