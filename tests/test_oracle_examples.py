"""The pages' worked examples, run through the oracle (fixtures under tests/golden/, each
citing its page and section). Logits are fed as ln p at T = 1 so that softmax recovers p."""
import numpy as np

import oracle
from _util import binom_z, chi2_pvalue, draw_from, golden, replicated_batch

N = 200_000


def _ln(p):
    return np.log(np.asarray(p, np.float64)).astype(np.float32)


def test_three_token_example():
    g = golden("three_token.txt")
    p, q = np.array(g["p"]), np.array(g["q"])
    # the fixture's own arithmetic: kept mass, gaps and totals as stated on the page
    np.testing.assert_allclose(np.minimum(q, p), g["min_qp"])
    np.testing.assert_allclose(np.maximum(p - q, 0), g["gap"], atol=1e-12)
    d = draw_from(q, N, seed=31)
    b = replicated_batch(np.stack([_ln(p), _ln(p)]), q[None, :], d[:, None], seed=301)
    o = oracle.run(b)
    acc = o["num_sampled"] == 2
    for tok, a in enumerate(g["accept_prob"]):
        sel = d == tok
        if a == 1.0:
            assert (~acc[sel]).sum() <= 2, "p/q >= 1 must (up to rounding) always accept"
        else:
            assert abs(binom_z(acc[sel].sum(), sel.sum(), a)) < 4.5
    assert abs(binom_z(acc.sum(), N, g["total_accept"][0])) < 4.5
    rejected_tokens = o["sampled"][~acc, 0]
    # a rejection always yields B: the residual has all its mass there
    assert np.sum(rejected_tokens != 1) <= 2
    first = np.bincount(o["sampled"][:, 0], minlength=3)
    assert chi2_pvalue(first, g["final"]) > 1e-3


def test_four_token_no_draft_probs_example():
    g = golden("four_token_no_draft_probs.txt")
    p = np.array(g["p"])
    dB = g["tokens"].index(g["draft"][0])
    b = replicated_batch(np.stack([_ln(p), _ln(p)]), None, np.full((N, 1), dB), seed=302)
    o = oracle.run(b)
    acc = o["num_sampled"] == 2
    assert abs(binom_z(acc.sum(), N, g["accept_prob"][0])) < 4.5
    rec = o["sampled"][~acc, 0]
    assert np.all(rec != dB)                                   # the rejected draft is excluded
    assert chi2_pvalue(np.bincount(rec, minlength=4), g["recovered"]) > 1e-3
    assert chi2_pvalue(np.bincount(o["sampled"][:, 0], minlength=4), g["final"]) > 1e-3


def test_four_token_bonus_example():
    g = golden("four_token_bonus.txt")
    B, C = (g["tokens"].index(t) for t in g["drafts"])
    p3 = np.array(g["p3"])
    uniform_q = np.full(4, 0.25)
    # case A: both drafts pass with certainty (p/q >= 1), so the bonus comes from p3
    p1 = np.array([0.1, 0.6, 0.2, 0.1])
    p2 = np.array([0.1, 0.1, 0.7, 0.1])
    b = replicated_batch(np.stack([_ln(p1), _ln(p2), _ln(p3)]), np.stack([uniform_q, uniform_q]),
                         np.tile([B, C], (N, 1)), seed=303)
    o = oracle.run(b)
    assert np.all(o["num_sampled"] == g["all_accepted_num_sampled"][0])
    assert np.all(o["sampled"][:, 0] == B) and np.all(o["sampled"][:, 1] == C)
    assert chi2_pvalue(np.bincount(o["sampled"][:, 2], minlength=4), p3) > 1e-3
    # case B: C is certainly rejected (p(C) ~ 1e-30, q(C) = 1): output B, recovered, no bonus
    p2b = np.array([0.3, 0.3, 1e-30, 0.4])
    q2b = np.array([0.0, 0.0, 1.0, 0.0])
    b = replicated_batch(np.stack([_ln(p1), _ln(p2b), _ln(p3)]), np.stack([uniform_q, q2b]),
                         np.tile([B, C], (N, 1)), seed=304)
    o = oracle.run(b)
    assert np.all(o["num_sampled"] == g["second_rejected_num_sampled"][0])
    assert np.all(o["sampled"][:, 2] == -1)
    assert np.all(o["num_rejected"] == 1)
    rec = np.bincount(o["sampled"][:, 1], minlength=4)
    assert chi2_pvalue(rec, np.maximum(p2b - q2b, 0)) > 1e-3


def test_five_token_example():
    g = golden("five_token.txt")
    p, q = np.array(g["p"]), np.array(g["q"])
    np.testing.assert_allclose(np.maximum(p - q, 0), g["residual_unnormalised"], atol=1e-12)
    np.testing.assert_allclose(np.maximum(p - q, 0).sum(), 1 - np.minimum(p, q).sum())
    d = g["tokens"].index(g["draft"][0])
    b = replicated_batch(np.stack([_ln(p), _ln(p)]), q[None, :], np.full((N, 1), d), seed=305)
    o = oracle.run(b)
    acc = o["num_sampled"] == 2
    assert abs(binom_z(acc.sum(), N, g["accept_prob"][0])) < 4.5
    rec = np.bincount(o["sampled"][~acc, 0], minlength=5)
    assert rec[0] == 0 and rec[4] == 0                         # p <= q: no residual mass
    assert chi2_pvalue(rec, g["residual"]) > 1e-3
