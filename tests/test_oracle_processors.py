"""Pins of the oracle's logits processors: the frequency penalty ([MTP-eagle] 其他 / 重复惩罚:
logit -= frequency_penalty * output_bin_counts) and the sampling constraints applied before the
target softmax ([spec-notes] 8.2 apply_logits_processors / apply_sampling_constraints;
[mini-sglang] "how tokens are sampled": top_k < 1 is the whole vocabulary, top_p in [1e-6, 1])."""
import os

import numpy as np
import pytest
from scipy import stats

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name), encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        k, v = line.split(None, 1)
        out[k] = float(v)
    return out


def _one_request(V, K, logits_rows, draft_ids, T=1.0, greedy=0, seed=3):
    b = workloads.make_batch(name="proc", data_seed=1, verify_seed=seed, K=[K], vocab_size=V,
                             logits_dtype="f32", q_mode="none", temperature=T,
                             greedy=np.array([greedy], np.uint8))
    b.logits = np.ascontiguousarray(logits_rows, np.float32)
    b.draft_ids = np.asarray(draft_ids, np.int32)
    return b


def test_frequency_penalty_worked_example():
    g = _golden("frequency_penalty.txt")
    V, the, cat = 300, int(g["token_the"]), int(g["token_cat"])
    row = np.zeros(V, np.float32)
    row[the], row[cat] = g["logit_the"], g["logit_cat"]
    for count, want in ((g["count_after_first"], g["penalised_the_after_first"]),
                        (g["count_after_second"], g["penalised_the_after_second"])):
        b = _one_request(V, 0, row[None, :], [], greedy=1)
        b.frequency_penalty = np.array([g["frequency_penalty"]], np.float32)
        counts = np.zeros((1, V), np.int32)
        counts[0, the] = int(count)
        b.output_bin_counts = counts
        r = oracle.run(b)
        # greedy: the row maximum is the penalised logit of "the" or "cat"'s 1.75
        assert r["row_max"][0] == max(np.float32(want), np.float32(g["logit_cat"]))
        assert r["sampled"][0, 0] == (the if want > g["logit_cat"] else cat)
    # without counts nothing changes
    b = _one_request(V, 0, row[None, :], [], greedy=1)
    b.frequency_penalty = np.array([0.5], np.float32)
    b.output_bin_counts = np.zeros((1, V), np.int32)
    assert oracle.run(b)["sampled"][0, 0] == the


def test_earlier_drafts_count_at_later_positions():
    """Row j conditions on drafts 0..j-1: a draft equal to v adds one to v's count there."""
    V = 64
    rows = np.zeros((3, V), np.float32)
    rows[:, 7] = 1.0
    rows[:, 9] = 0.8
    b = _one_request(V, 2, rows, [7, 7], greedy=1)
    b.frequency_penalty = np.array([0.25], np.float32)
    b.output_bin_counts = np.zeros((1, V), np.int32)
    r = oracle.run(b)
    # row 0: 7 (1.0); row 1: 7 counted once -> 0.75 < 0.8: argmax 9; row 2: 7 twice -> 0.5
    assert list(r["row_argmax"]) == [7, 9, 9]
    assert r["num_sampled"][0] == 2 and list(r["sampled"][0]) == [7, 9, -1]


def test_counts_row_mapping_and_negative_penalty():
    V = 32
    row = np.linspace(0, 1, V, dtype=np.float32)
    counts = np.zeros((3, V), np.int32)
    counts[2, 0] = 4
    b = _one_request(V, 0, row[None, :], [], greedy=1)
    b.frequency_penalty = np.array([-0.5], np.float32)      # a negative penalty favours token 0
    b.output_bin_counts = counts
    b.counts_row = np.array([2], np.int32)
    r = oracle.run(b)
    assert r["sampled"][0, 0] == 0 and r["row_max"][0] == np.float32(2.0)


def _brute_select(x, k, p):
    """Independent restatement: sort, top-k by rank with ties kept, top-p over groups of
    equal values by the mass strictly above, in float64."""
    x = np.asarray(x, np.float64)
    V = x.size
    keep = np.ones(V, bool)
    if 1 <= k < V:
        kth = np.sort(x)[::-1][k - 1]
        keep &= x >= kth
    if p < 1:
        p = max(p, 1e-6)
        m = x.max()
        t = np.array([oracle.exp32(np.float32(v - m)) for v in x.astype(np.float32)], np.float64)
        Z = t[keep].sum()
        kept = np.zeros(V, bool)
        for val in np.unique(x[keep])[::-1]:
            above = t[keep & (x > val)].sum()
            if above < p * Z:
                kept |= keep & (x == val)
            else:
                break
        keep = kept
    return keep


@pytest.mark.parametrize("seed", range(8))
def test_selection_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(5, 300))
    x = np.round(rng.normal(0, 2, V) * 4) / 4                   # many ties
    x = x.astype(np.float32)
    for k, p in ((0, 1.0), (5, 1.0), (1, 1.0), (V - 1, 1.0), (0, 0.9), (0, 0.5), (7, 0.8),
                 (0, 1e-9), (3, 0.999), (V, 0.3)):
        tau, Sk, margin = oracle.select_row(x, k, p)
        keep = _brute_select(x, k, p)
        assert np.array_equal(x >= tau, keep), (k, p)
        m = x.max()
        want = sum(float(oracle.exp32(np.float32(v - m))) for v in x[keep])
        assert Sk == pytest.approx(want, rel=1e-12)
        if p >= 1:
            assert margin == np.inf


def test_top_p_margin_is_the_distance_to_the_boundary():
    x = np.log(np.array([0.5, 0.3, 0.2], np.float64)).astype(np.float32)
    tau, Sk, margin = oracle.select_row(x, 0, 0.8)
    # masses strictly above: 0, 0.5, 0.8: the third token sits on the boundary (either side)
    assert tau in (x[1], x[2])
    assert margin < 1e-6
    tau, _, margin = oracle.select_row(x, 0, 0.65)
    assert tau == x[1] and margin == pytest.approx(0.15, abs=1e-6)


def test_top_k_one_is_greedy():
    b = workloads.workload(1)
    b.top_k = np.ones(b.num_reqs, np.int32)
    r = oracle.run(b)
    for i in range(b.num_reqs):
        js = r["num_sampled"][i] - 1
        assert r["sampled"][i, js] == r["row_argmax"][b.cu_num_draft[i] + i + js]


@pytest.mark.parametrize("k,p", [(4, 1.0), (0, 0.7), (6, 0.8)])
def test_outputs_follow_the_constrained_target(k, p):
    """Losslessness with processors: with a draft distribution q the emitted token of position 0
    follows p' (p under the constraints, renormalised), not p."""
    V, n = 10, 12000
    row = np.linspace(1.0, -1.0, V).astype(np.float32)
    b = workloads.make_batch(name="law", data_seed=2, verify_seed=17, K=[1] * n, vocab_size=V,
                             logits_dtype="f32", q_mode="noisy", q_noise=1.0, temperature=1.0)
    b.logits = np.tile(row, (b.num_rows, 1))
    q = np.full(V, 1.0 / V, np.float32)
    b.draft_probs = np.tile(q, (n, 1))
    b.draft_ids = np.random.default_rng(4).integers(0, V, n).astype(np.int32)
    b.top_k = np.full(n, k, np.int32)
    b.top_p = np.full(n, p, np.float32)
    r = oracle.run(b)
    tok = r["sampled"][:, 0]
    keep = _brute_select(row, k, p)
    pp = np.where(keep, np.exp(row.astype(np.float64) - row.max()), 0.0)
    pp /= pp.sum()
    counts = np.bincount(tok, minlength=V)
    assert np.all(counts[~keep] == 0)
    assert stats.chisquare(counts[keep], pp[keep] * n).pvalue > 1e-4


def test_constraints_do_not_touch_greedy_requests_and_the_max_is_always_kept():
    b = workloads.workload(1)
    base = oracle.run(b)
    b.top_p = np.full(b.num_reqs, 1e-9, np.float32)               # only the max survives
    r = oracle.run(b)
    g = b.is_greedy != 0
    assert np.array_equal(r["sampled"][g], base["sampled"][g])
    logits = (b.logits.astype(np.uint32) << 16).view(np.float32)
    for i in np.flatnonzero(~g):
        js = r["num_sampled"][i] - 1
        row = b.cu_num_draft[i] + i + js
        tok = r["sampled"][i, js]
        x = np.float32(logits[row, tok]) * np.float32(np.float32(1.0) / b.temperature[i])
        assert x == r["row_max"][row]                              # a token of the maximum


def test_large_and_negative_counts():
    """The count enters the one-rounding fma as a binary32 value (rounded to nearest): 2^24 + 1
    becomes 2^24, so a token with that count ties one with count 2^24 and the lower index wins;
    with the count taken exactly it would lose by 2^-20. A negative count raises the logit."""
    V = 64
    row = np.full(V, -5.0, np.float32)
    row[3] = row[9] = 16.0
    b = _one_request(V, 0, row[None, :], [], greedy=1)
    b.frequency_penalty = np.array([2.0 ** -20], np.float32)
    counts = np.zeros((1, V), np.int32)
    counts[0, 3] = (1 << 24) + 1
    counts[0, 9] = 1 << 24
    b.output_bin_counts = counts
    r = oracle.run(b)
    assert r["row_max"][0] == np.float32(0.0)     # 16 - 2^-20 * 2^24 for both tokens
    assert r["sampled"][0, 0] == 3                # a tie: the lower index

    row = np.zeros(V, np.float32)
    row[5], row[7] = 2.0, 1.0
    b = _one_request(V, 0, row[None, :], [], greedy=1)
    b.frequency_penalty = np.array([0.5], np.float32)
    counts = np.zeros((1, V), np.int32)
    counts[0, 7] = -3                              # 1 + 0.5 * 3 = 2.5 > 2
    b.output_bin_counts = counts
    r = oracle.run(b)
    assert r["row_max"][0] == np.float32(2.5)
    assert r["sampled"][0, 0] == 7
