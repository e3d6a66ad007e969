"""Pins of the oracle's binary64 race noise (the fp64 Gumbel option, [spec-in-vllm] 7.3:
use_fp64_gumbel draws the race noise in double precision).

What each test ties the oracle to:
  - the 52-bit uniform: its definition evaluated with exact integer arithmetic;
  - the binary64 log: mpmath at 120 bits, correctly rounded (at most 2 ulp apart);
  - the clock layout: clocks recomputed in float64 from Philox words that the Triton
    library's own Philox routine produces (Triton interpreter on the CPU);
  - the clock law: i.i.d. Exp(1) by KS and chi-square tests, as for the binary32 clocks;
  - the race: the empirical output law equals p (and the renormalised residual), and every
    winner equals a float64 brute force from the oracle's own clocks;
  - the option changes nothing but the races: acceptance decisions and greedy outputs are
    those of the binary32 mode.
"""
import numpy as np
import pytest
from scipy import stats

import oracle
import workloads
from _util import chi2_pvalue, draw_from, replicated_batch
from test_oracle_rng import _triton_philox

mpmath = pytest.importorskip("mpmath")


def _u64_exact(hi, lo):
    m = (int(hi) << 20) | (int(lo) >> 12)
    return (m + 0.5) / 2.0**52                       # exact: m + 1/2 has 53 significant bits


def test_uniform64_extremes_and_exactness():
    assert oracle.uniform64(0, 0) == 2.0**-53
    assert oracle.uniform64(0xFFFFFFFF, 0xFFFFFFFF) == 1.0 - 2.0**-53
    assert oracle.uniform64(0, 0xFFF) == 2.0**-53          # low 12 bits of the second word drop
    assert oracle.uniform64(0, 0x1000) == 3 * 2.0**-53
    assert oracle.uniform64(1, 0) == (2**20 + 0.5) / 2.0**52
    rng = np.random.default_rng(5)
    for hi, lo in rng.integers(0, 2**32, (500, 2), dtype=np.uint64):
        u = oracle.uniform64(int(hi), int(lo))
        assert 0.0 < u < 1.0 and u == _u64_exact(hi, lo)
    # neighbouring 52-bit codes are 2^-52 apart: 29 more bits than the binary32 uniform
    assert oracle.uniform64(7, 0x2000) - oracle.uniform64(7, 0x1000) == 2.0**-52


def _ulps(a, b):
    ia = np.array([a], np.float64).view(np.int64)[0]
    ib = np.array([b], np.float64).view(np.int64)[0]
    return abs(int(ia) - int(ib))


def test_log64_against_mpmath():
    mpmath.mp.prec = 120
    rng = np.random.default_rng(11)
    xs = [_u64_exact(h, l) for h, l in rng.integers(0, 2**32, (1500, 2), dtype=np.uint64)]
    xs += [1.0 - k * 2.0**-53 for k in range(1, 120)] + [1.0 + k * 2.0**-52 for k in range(1, 120)]
    xs += list(np.exp(rng.uniform(np.log(1e-300), np.log(1e300), 1500)))
    xs += [2.0**-53, 2.0**-52, 0.5, 2.0, np.sqrt(0.5), np.sqrt(2.0), np.nextafter(np.sqrt(2.0), 3),
           np.nextafter(np.sqrt(2.0), 0), 5e-324, 2.0**-1030, 2.2250738585072014e-308,
           np.nextafter(2.2250738585072014e-308, 0), 1.7976931348623157e308]
    worst = 0
    for x in xs:
        want = float(mpmath.log(mpmath.mpf(float(x))))
        got = oracle.log64(float(x))
        worst = max(worst, _ulps(got, want))
    assert worst <= 2, worst
    assert oracle.log64(1.0) == 0.0
    assert oracle.log64(0.0) == -np.inf and oracle.log64(np.inf) == np.inf
    assert np.isnan(oracle.log64(-1.0)) and np.isnan(oracle.log64(np.nan))
    # the array entry point is the same function
    arr = np.array(xs[:300])
    np.testing.assert_array_equal(oracle.log64_n(arr), [oracle.log64(float(x)) for x in arr])


def test_largest_clock_is_beyond_the_binary32_cap():
    """The largest value -log U can take: 53 ln 2 = 36.74 with 52-bit uniforms, against
    24 ln 2 = 16.64 with the binary32 ones (the truncated tail the option removes)."""
    mpmath.mp.prec = 120
    top64 = -oracle.log64(oracle.uniform64(0, 0))
    top32 = -oracle.log32(oracle.uniform_from_word(0))
    assert top64 == pytest.approx(float(53 * mpmath.log(2)), rel=1e-15)
    assert top32 == pytest.approx(float(24 * mpmath.log(2)), rel=1e-6)
    small64 = -oracle.log64(oracle.uniform64(0xFFFFFFFF, 0xFFFFFFFF))
    assert small64 == pytest.approx(2.0**-53, rel=1e-12)    # smallest positive excess


def test_clock64_layout_matches_triton(tmp_path):
    """Token v (group g = v >> 6, slot s = v & 63) at (request i, position j): counter
    (g, j, i, 32) gives W from words 0 and 1 and the argmin slot a = word 2 & 63,
    E_min = -ln(W) / 64; slot s != a adds -ln U_s, U_s from words (0, 1) for even s and (2, 3)
    for odd s of counter (g, j, i, 33 + s // 2)."""
    seed, j, i = 0xC0FFEE0012345678, 2, 9
    groups = [(0, 3), (7, 8)]                        # 33 calls per group; 128 counters a request
    reqs = []
    for gs in groups:
        ctr = np.array([[g, j, i, 32 + k] for g in gs for k in range(33)], dtype=np.uint32)
        reqs.append((seed, np.vstack([ctr, np.zeros((128 - ctr.shape[0], 4), np.uint32)])))
    words = _triton_philox(reqs, tmp_path)
    checked = 0
    for gs, w in zip(groups, words):
        for k, g in enumerate(gs):
            head = w[33 * k]
            emin = -np.log(_u64_exact(head[0], head[1])) / 64.0
            a = int(head[2]) & 63
            want = np.empty(64)
            for s_ in range(64):
                call = w[33 * k + 1 + s_ // 2]
                h = 2 * (s_ & 1)
                want[s_] = emin if s_ == a else emin - np.log(_u64_exact(call[h], call[h + 1]))
            got = oracle.race_clocks64(seed, j, i, 64 * (g + 1))[64 * g:]
            np.testing.assert_allclose(got, want, rtol=1e-13, atol=0)
            checked += 64
    assert checked == 256


def test_clocks64_are_iid_exponential():
    n = 64 * 10_000
    e = oracle.race_clocks64(2024, 1, 5, n)
    assert stats.kstest(e, "expon").pvalue > 1e-3
    blocks = e.reshape(-1, 64)
    for s_ in (0, 1, 30, 63):
        assert stats.kstest(blocks[:, s_], "expon").pvalue > 1e-3
    argmin = np.bincount(blocks.argmin(axis=1), minlength=64)
    assert stats.chisquare(argmin).pvalue > 1e-3
    assert stats.kstest(blocks.min(axis=1) * 64, "expon").pvalue > 1e-3
    assert abs(np.corrcoef(blocks[:, 2], blocks[:, 3])[0, 1]) < 0.02   # slots of one call
    other = oracle.race_clocks64(2024, 2, 5, 64 * 1250)
    assert abs(np.corrcoef(e[: other.size], other)[0, 1]) < 0.03
    e32 = oracle.race_clocks(2024, 1, 5, 64 * 1250).astype(np.float64)  # a separate stream
    assert abs(np.corrcoef(e[: e32.size], e32)[0, 1]) < 0.03


def _softmax(x, T=1.0):
    z = np.asarray(x, np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


N = 200_000


@pytest.mark.parametrize("V,T", [(3, 1.0), (8, 0.8), (16, 1.2)])
def test_fp64_race_is_lossless(V, T):
    K = 2
    rng = np.random.default_rng(900 + V)
    logits = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    q = np.stack([_softmax(logits[j] + rng.standard_normal(V)) for j in range(K)]).astype(np.float32)
    d = np.stack([draw_from(q[j], N, seed=910 + 10 * V + j) for j in range(K)], axis=1)
    b = replicated_batch(logits, q, d, temperature=T, seed=920 + V)
    b.fp64_gumbel = True
    o = oracle.run(b)
    s = o["sampled"]
    p = [_softmax(logits[j], T) for j in range(K + 1)]
    assert chi2_pvalue(np.bincount(s[:, 0], minlength=V), p[0]) > 1e-3
    sel = o["num_sampled"] == 3
    assert chi2_pvalue(np.bincount(s[sel, 2], minlength=V), p[2]) > 1e-3
    # the token at a rejection of position 0 ~ the residual max(0, p - q) renormalised
    rej = o["num_sampled"] == 1
    r = np.maximum(p[0] - q[0].astype(np.float64), 0)
    assert chi2_pvalue(np.bincount(s[rej, 0], minlength=V), r / r.sum()) > 1e-3


def test_fp64_gumbel_max_and_exclusion_are_lossless():
    V = 12
    rng = np.random.default_rng(31)
    row = (rng.standard_normal((1, V)) * 2).astype(np.float32)
    b = replicated_batch(row, None, np.zeros((N, 0), np.int32), temperature=0.7, seed=32)
    b.fp64_gumbel = True
    o = oracle.run(b)
    assert chi2_pvalue(np.bincount(o["sampled"][:, 0], minlength=V), _softmax(row[0], 0.7)) > 1e-3
    rows = (rng.standard_normal((2, V)) * 2).astype(np.float32)
    d = np.full((N, 1), int(np.argmax(rows[0])), np.int32)     # draft ids only, mostly rejected
    b = replicated_batch(rows, None, d, seed=33)
    b.fp64_gumbel = True
    o = oracle.run(b)
    rej = o["num_sampled"] == 1
    p = _softmax(rows[0])
    p[d[0, 0]] = 0.0                                            # p without the rejected draft
    assert chi2_pvalue(np.bincount(o["sampled"][rej, 0], minlength=V), p / p.sum()) > 1e-3


def test_fp64_race_winner_brute_force():
    """Every race winner equals the argmax of log w_v - log E_v computed in float64 from the
    oracle's binary64 clocks (p-race, residual race, exclusion race; a request index base)."""
    rng = np.random.default_rng(77)
    base, checked = 3, 0
    for trial in range(240):
        V = int(rng.integers(2, 300))
        mode = trial % 3                       # 0 bonus, 1 residual, 2 exclusion
        K = 1
        logits = (rng.standard_normal((3 + K, V)) * 2).astype(np.float32)
        q = None
        if mode == 1:
            q = (rng.random((1 + K, V)).astype(np.float32) ** 3)
            q /= q.sum(1, keepdims=True)
        d = rng.integers(0, V, 1 + K).astype(np.int32)
        js = 1 if mode == 0 else 0
        u = np.float32([0.0, 0.0 if mode == 0 else 1e30])
        b = workloads.Batch(name="bf", logits=logits, logits_dtype="f32", vocab_size=V,
                            draft_ids=d, draft_probs=q, cu_num_draft=np.array([0, 1, 2], np.int32),
                            temperature=np.ones(2, np.float32), is_greedy=np.zeros(2, np.uint8),
                            seed=5000 + trial, fp64_gumbel=True)
        o = oracle.run(b, u_override=u, req_index_base=base)
        assert o["jstar"][1] == js
        row = 2 + js                            # rows of request 1 start at cu[1] + 1 = 2
        x = logits[row].astype(np.float64)
        logp = x - x.max() - np.log(np.exp(x - x.max()).sum())
        g = -np.log(oracle.race_clocks64(5000 + trial, js, base + 1, V))
        if mode == 1:
            w = np.maximum(np.exp(logp) - q[1].astype(np.float64), 0)
            keys = np.where(w > 0, np.log(np.where(w > 0, w, 1)) + g, -np.inf)
        else:
            keys = logp + g
            if mode == 2:
                keys[d[1]] = -np.inf
        order = np.argsort(-keys, kind="stable")
        if np.isfinite(keys[order[1]]) and keys[order[0]] - keys[order[1]] < 1e-6:
            continue                            # too close to call in another precision
        assert o["sampled"][1, js] == order[0], (trial, mode)
        checked += 1
    assert checked > 200


@pytest.mark.parametrize("c", [1, 2])
def test_fp64_option_changes_only_the_races(c):
    b = workloads.workload(c, num_reqs=48)
    o32 = oracle.run(b)
    b.fp64_gumbel = True
    o64 = oracle.run(b)
    np.testing.assert_array_equal(o64["jstar"], o32["jstar"])
    np.testing.assert_array_equal(o64["accept_margin"], o32["accept_margin"])
    for k in ("row_max", "row_sumexp", "row_argmax", "num_sampled", "num_rejected"):
        np.testing.assert_array_equal(o64[k], o32[k])
    greedy = (b.is_greedy != 0) | ~(b.temperature > 0)
    np.testing.assert_array_equal(o64["sampled"][greedy], o32["sampled"][greedy])
    differ = (o64["sampled"] != o32["sampled"]).any(axis=1)
    assert differ[~greedy].mean() > 0.5        # an independent noise stream for the races
