"""Pins of the oracle's synthetic acceptance mode ([spec-in-vllm] 7.2: preset per-position
rates, or a target mean length turned into minimum-variance rates; 7.4: the rejection kernel
compares with the rate) and of the chunked-prefill count correction ([MTP-eagle]
get_num_sampled_and_rejected)."""
import itertools

import numpy as np
import pytest
from scipy import stats

import oracle
import workloads


def _var_of_rates(a):
    """Variance of the accepted count N when P(N > j) = a_j."""
    a = np.concatenate([[1.0], np.asarray(a, np.float64), [0.0]])
    pk = a[:-1] - a[1:]                      # P(N = k), k = 0..K
    k = np.arange(pk.size)
    mean = (k * pk).sum()
    return (k * k * pk).sum() - mean * mean, mean


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_length_rates_have_the_least_variance(K):
    """Brute force over every non-increasing rate vector on a 0.1 grid with the same mean."""
    grid = np.round(np.arange(0, 11) / 10.0, 10)
    best = {}
    for vec in itertools.product(grid, repeat=K):
        if any(vec[i] < vec[i + 1] for i in range(K - 1)):
            continue
        var, mean = _var_of_rates(vec)
        key = round(mean, 6)
        best[key] = min(best.get(key, np.inf), var)
    for mean_acc, vmin in best.items():
        r = oracle.synthetic_rates(1.0 + mean_acc, K)
        assert np.all((r >= 0) & (r <= 1)) and np.all(np.diff(r) <= 0)
        var, mean = _var_of_rates(r)
        assert mean == pytest.approx(mean_acc, abs=1e-6)
        assert var <= vmin + 1e-6
        f = mean_acc - np.floor(mean_acc)
        assert var == pytest.approx(f * (1 - f), abs=1e-6)       # two-point law


def test_length_rates_range():
    assert np.array_equal(oracle.synthetic_rates(1.0, 3), [0, 0, 0])
    assert np.array_equal(oracle.synthetic_rates(4.0, 3), [1, 1, 1])
    for bad in (0.99, 4.01, float("nan")):
        with pytest.raises(ValueError):
            oracle.synthetic_rates(bad, 3)


def _batch(n, K, V, seed, **kw):
    rng = np.random.default_rng(seed)
    return workloads.make_batch(name="syn", data_seed=seed, verify_seed=seed + 11, K=[K] * n,
                                vocab_size=V, logits_dtype="f32", sigma=1.5, q_mode="none",
                                p_argmax=0.3, temperature=rng.uniform(0.5, 1.5, n).astype(np.float32),
                                **kw)


def test_acceptance_follows_the_unconditional_rates():
    rates = np.array([0.9, 0.6, 0.6, 0.1], np.float32)
    b = _batch(4000, 4, 16, 5)
    b.synthetic_rates = rates
    r = oracle.run(b)
    acc = r["num_sampled"] - 1
    n = acc.size
    for j, a in enumerate(rates):
        frac = float(np.mean(acc > j))
        assert abs(frac - a) <= 5 * np.sqrt(a * (1 - a) / n) + 1e-9, (j, frac, a)
    assert np.all(r["num_rejected"] == 4 - acc)


def test_target_length_gives_the_mean_length():
    b = _batch(4000, 5, 16, 6)
    b.synthetic_rates = oracle.synthetic_rates(3.4, 5)            # accept 2 or 3 drafts
    r = oracle.run(b)
    acc = r["num_sampled"] - 1
    assert set(np.unique(acc)) <= {2, 3}
    assert abs(acc.mean() - 2.4) < 5 * np.sqrt(0.24 / acc.size)


def test_conditional_rule_with_given_uniforms():
    """Position j is accepted iff a_j / a_{j-1} >= u_j (binary32), whatever p and q are."""
    rates = np.array([0.8, 0.4, 0.4, 0.0], np.float32)
    c = [np.float32(0.8), np.float32(0.4) / np.float32(0.8), np.float32(1.0), np.float32(0.0)]
    b = _batch(200, 4, 32, 7, greedy=(np.arange(200) % 3 == 0).astype(np.uint8))
    b.synthetic_rates = rates
    u = np.random.default_rng(8).random(b.num_draft_tokens).astype(np.float32)
    u = np.clip(u, 1e-6, 1 - 1e-6)
    r = oracle.run(b, u_override=u)
    for i in range(b.num_reqs):
        js = next((j for j in range(4) if not (c[j] >= u[4 * i + j])), 4)
        assert r["num_sampled"][i] == js + 1
        assert np.array_equal(r["sampled"][i, :js], b.draft_ids[4 * i:4 * i + js])


def test_token_at_the_first_rejection_is_a_draw_from_p():
    V, n = 12, 6000
    b = _batch(n, 2, V, 9)
    row = np.linspace(-2.0, 2.0, V).astype(np.float32)
    b.logits = np.tile(row, (b.num_rows, 1))
    b.temperature[:] = 1.0
    b.synthetic_rates = np.array([0.5, 0.2], np.float32)
    r = oracle.run(b)
    js = r["num_sampled"] - 1
    tok = r["sampled"][np.arange(n), js]
    p = np.exp(row.astype(np.float64) - row.max())
    p /= p.sum()
    counts = np.bincount(tok, minlength=V)
    assert stats.chisquare(counts, p * n).pvalue > 1e-4
    assert np.all(r["race_kind"] == oracle.RACE_TARGET)


def test_greedy_requests_emit_the_argmax_and_invalid_ids_are_rejected():
    b = _batch(300, 3, 40, 10, greedy=np.ones(300, np.uint8))
    b.synthetic_rates = np.array([1.0, 1.0, 1.0], np.float32)
    b.draft_ids[3 * 7 + 1] = 40                                    # request 7, position 1
    b.draft_ids[3 * 9] = -1                                        # request 9, position 0
    r = oracle.run(b)
    for i in range(b.num_reqs):
        js = r["num_sampled"][i] - 1
        want = 1 if i == 7 else (0 if i == 9 else 3)
        assert js == want
        assert r["sampled"][i, js] == r["row_argmax"][b.cu_num_draft[i] + i + js]


def test_partial_prefill_requests_report_nothing():
    b = workloads.workload(1)
    full = oracle.run(b)
    b.partial_prefill = np.zeros(b.num_reqs, np.uint8)
    b.partial_prefill[[0, 5, 17, 63]] = 1
    part = oracle.run(b)
    for i in range(b.num_reqs):
        if b.partial_prefill[i]:
            assert part["num_sampled"][i] == 0 and part["num_rejected"][i] == 0
            assert np.all(part["sampled"][i] == -1)
        else:
            assert np.array_equal(part["sampled"][i], full["sampled"][i])
            assert part["num_sampled"][i] == full["num_sampled"][i]
            assert part["num_rejected"][i] == full["num_rejected"][i]
    for k in ("row_max", "row_sumexp", "row_argmax"):
        assert np.array_equal(part[k], full[k])
