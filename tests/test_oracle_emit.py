"""Structural pins of the oracle: the per-request scan and emit, greedy rules, invalid ids,
inconsistent batches, keyed-RNG invariances, and a brute-force check of the race winner."""
import itertools

import numpy as np
import pytest

import oracle
from _util import replicated_batch
from workloads import Batch


def _batch(logits, q, ids, cu, T, greedy, seed=5, dtype="f32"):
    n = len(cu) - 1
    return Batch(name="t", logits=np.ascontiguousarray(logits), logits_dtype=dtype,
                 vocab_size=logits.shape[1], draft_ids=np.asarray(ids, np.int32),
                 draft_probs=None if q is None else np.ascontiguousarray(q, np.float32),
                 cu_num_draft=np.asarray(cu, np.int32),
                 temperature=np.broadcast_to(np.float32(T), (n,)).copy(),
                 is_greedy=np.broadcast_to(np.uint8(greedy), (n,)).copy(), seed=seed)


@pytest.mark.parametrize("with_q", [False, True])
def test_forced_accept_patterns(with_q):
    """Every accept/reject pattern for K = 0..4 (uniforms overridden: 0 accepts, 1e30 rejects):
    slots before j* hold the drafts, slot j* the recovered or bonus token, the rest -1."""
    V = 16
    rng = np.random.default_rng(3)
    pats = [(K, bits) for K in range(5) for bits in itertools.product([0, 1], repeat=K)]
    Ks = [K for K, _ in pats]
    cu = np.concatenate([[0], np.cumsum(Ks)]).astype(np.int32)
    R = int(cu[-1]) + len(Ks)
    logits = (rng.standard_normal((R, V)) * 2).astype(np.float32)
    ids = rng.integers(0, V, int(cu[-1])).astype(np.int32)
    q = None
    if with_q:
        q = rng.random((int(cu[-1]), V)).astype(np.float32) + 0.01
        q /= q.sum(1, keepdims=True)
    u = np.concatenate([[0.0 if b == 0 else 1e30 for b in bits] for _, bits in pats] or [[]])
    b = _batch(logits, q, ids, cu, 1.0, 0)
    o = oracle.run(b, u_override=u.astype(np.float32))
    for i, (K, bits) in enumerate(pats):
        js = next((j for j, bt in enumerate(bits) if bt), K)
        row = o["sampled"][i]
        assert o["jstar"][i] == js
        assert list(row[:js]) == list(ids[cu[i]:cu[i] + js])
        assert 0 <= row[js] < V
        assert np.all(row[js + 1:] == -1)
        assert o["num_sampled"][i] == js + 1 and o["num_rejected"][i] == K - js
        if js < K and not with_q:
            assert row[js] != ids[cu[i] + js]
        kind = o["race_kind"][i]
        assert kind == (oracle.RACE_BONUS if js == K else
                        (oracle.RACE_RESIDUAL if with_q else oracle.RACE_EXCLUDE))


def test_zero_temperature_and_nan_are_greedy():
    V = 10
    rng = np.random.default_rng(4)
    logits = (rng.standard_normal((6, V)) * 2).astype(np.float32)
    amax = logits.argmax(1)
    ids = np.array([amax[0], (amax[1] + 1) % V, amax[3], amax[4]], np.int32)
    b = _batch(logits, None, ids, [0, 2, 4], 0.0, 0)
    b.temperature[1] = np.nan
    o = oracle.run(b)
    np.testing.assert_array_equal(o["sampled"][0], [amax[0], amax[1], -1])
    np.testing.assert_array_equal(o["sampled"][1], [amax[3], amax[4], amax[5]])


def test_out_of_range_draft_ids_are_rejected():
    V = 12
    rng = np.random.default_rng(5)
    logits = (rng.standard_normal((4, V))).astype(np.float32)
    for bad in (-1, V, 2**31 - 1):
        for q in (None, np.full((2, V), 1.0 / V, np.float32)):
            b = _batch(logits, q, [bad, 0], [0, 2], 1.0, 0)
            o = oracle.run(b)
            assert o["num_sampled"][0] == 1 and o["num_rejected"][0] == 2
            assert 0 <= o["sampled"][0, 0] < V
            assert np.isinf(o["accept_margin"][0])


def test_zero_draft_probability_is_rejected():
    V = 6
    logits = np.zeros((2, V), np.float32)
    q = np.full((1, V), 0.2, np.float32)
    q[0, 3] = 0.0
    o = oracle.run(_batch(logits, q, [3], [0, 1], 1.0, 0), u_override=np.float32([0.0]))
    assert o["num_sampled"][0] == 1                            # even with u = 0


def test_inconsistent_batches_emit_nothing():
    logits = np.zeros((5, 4), np.float32)
    b = _batch(logits, None, [0, 1, 2], [0, 3, 2], 1.0, 0)     # decreasing prefix sum
    o = oracle.run(b)
    assert o["status"] == oracle.EBATCH
    assert np.all(o["num_sampled"] == 0) and np.all(o["sampled"] == -1)
    b = _batch(logits[:4], None, [0, 1, 2], [0, 3], 1.0, 0)
    o = oracle.run(b, max_spec_len=2)                          # K above the stated maximum
    assert o["status"] == oracle.EBATCH


def test_sharding_by_requests_with_index_base_reproduces_the_batch():
    import workloads
    b = workloads.make_batch(name="s", data_seed=3, verify_seed=77, K=[3, 0, 2, 5, 1, 4, 3, 2],
                             vocab_size=257, logits_dtype="bf16", sigma=2.0, q_mode="noisy",
                             q_noise=1.0, temperature=0.9)
    full = oracle.run(b, max_spec_len=5)
    cu = b.cu_num_draft
    for cut in (1, 3, 6):
        parts = []
        for lo, hi in ((0, cut), (cut, b.num_reqs)):
            r0, r1 = cu[lo] + lo, cu[hi] + hi
            sub = Batch(name="part", logits=b.logits[r0:r1], logits_dtype="bf16", vocab_size=257,
                        draft_ids=b.draft_ids[cu[lo]:cu[hi]],
                        draft_probs=b.draft_probs[cu[lo]:cu[hi]],
                        cu_num_draft=(cu[lo:hi + 1] - cu[lo]).astype(np.int32),
                        temperature=b.temperature[lo:hi], is_greedy=b.is_greedy[lo:hi], seed=77)
            parts.append(oracle.run(sub, max_spec_len=5, req_index_base=lo))
        for k in ("sampled", "num_sampled", "num_rejected"):
            np.testing.assert_array_equal(np.concatenate([p[k] for p in parts]), full[k])
    again = oracle.run(b, max_spec_len=5)
    np.testing.assert_array_equal(again["sampled"], full["sampled"])
    other = oracle.run(b, max_spec_len=5, seed=78)
    assert not np.array_equal(other["sampled"], full["sampled"])


def test_race_winner_brute_force():
    """Recompute every race key in float64 from the race clocks of (request, position) and compare
    the winner. Races run at positions 0..2 of the second request of a batch, with a request
    index base, so the counter's position and request words are both exercised."""
    rng = np.random.default_rng(17)
    checked = 0
    base = 5
    for trial in range(300):
        V = int(rng.integers(2, 40))
        T = float(rng.choice([1.0, 0.5, 1.7]))
        mode = trial % 3                       # 0 bonus, 1 residual, 2 exclusion
        K = int(rng.integers(0, 3)) if mode == 0 else int(rng.integers(1, 3))
        js = K if mode == 0 else int(rng.integers(0, K))      # position of the race
        Kt = [1, K]                                            # request 0 is a bystander
        cu = [0, 1, 1 + K]
        R = 1 + K + 2
        logits = (rng.standard_normal((R, V)) * 2).astype(np.float32)
        q = None
        if mode == 1:
            q = (rng.random((1 + K, V)).astype(np.float32) ** 3)
            q /= q.sum(1, keepdims=True)
        d = rng.integers(0, V, 1 + K).astype(np.int32)
        u = np.float32([0.0] + [0.0 if j < js else 1e30 for j in range(K)])
        seed = 1000 + trial
        b = _batch(logits, q, d, cu, T, 0, seed=seed)
        o = oracle.run(b, u_override=u, req_index_base=base)
        assert o["jstar"][1] == js
        tok = int(o["sampled"][1, js])
        invT = np.float32(1.0) / np.float32(T)
        row = cu[1] + 1 + js
        x = (logits[row] * invT).astype(np.float64)
        clocks = oracle.race_clocks(seed, js, base + 1, V).astype(np.float64)
        g = -np.log(clocks)
        if mode == 1:
            p = np.exp(x - x.max()) / np.exp(x - x.max()).sum()
            w = np.maximum(p - q[cu[1] + js].astype(np.float64), 0)
            keys = np.where(w > 0, np.log(np.where(w > 0, w, 1)) + g, -np.inf)
        else:
            keys = x + g
            if mode == 2:
                keys[d[cu[1] + js]] = -np.inf
        order = np.argsort(-keys, kind="stable")
        if V > 1 and np.isfinite(keys[order[1]]) and keys[order[0]] - keys[order[1]] < 1e-4:
            continue                           # too close to call in another precision
        assert tok == order[0], (trial, mode, tok, order[:3])
        checked += 1
    assert checked > 250
