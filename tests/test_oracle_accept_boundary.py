"""Pins of the oracle's acceptance comparison at its exact boundary.

The test of draft d is p(d) / q(d) >= u in binary32 ([spec-notes] NO_DRAFT_PROBS answer code:
accept when draft_prob > 0 and target_prob / draft_prob >= uniform). Statistical pins cannot
tell >= from >, nor a quotient rounded in binary32 from one taken in double: both differ on a
set of uniforms of measure zero. Here the uniform is overridden with the binary32 quotient
itself, and with its neighbours one ulp away.

The rows are built so that p(d) is known without the oracle: n tokens share the largest logit
and every other token is -inf, so exp(x_d - m) = exp(0) = 1, S = n and p(d) = fl(1 / n). The
expected quotient fl(p(d) / q(d)) comes from numpy's IEEE binary32 division, not from the
oracle's code.
"""
import numpy as np
import pytest

import oracle
from workloads import Batch

F32 = np.float32


def _rows(V, n, dtype):
    """One request, K = 1: row 0 with n tokens at logit 0 (token 0 among them) and the rest
    -inf; the bonus row is flat."""
    r = np.full((2, V), -np.inf, np.float32)
    r[0, :n] = 0.0
    r[1, :] = 0.0
    if dtype == "bf16":
        return (r.view(np.uint32) >> 16).astype(np.uint16)     # 0 and -inf are exact in bf16
    return r


def _run(V, n, q_d, u, dtype="f32", d=0):
    q = None
    if q_d is not None:
        q = np.full((1, V), (1.0 - q_d) / max(V - 1, 1), np.float32)
        q[0, d] = q_d
    b = Batch(name="boundary", logits=_rows(V, n, dtype), logits_dtype=dtype, vocab_size=V,
              draft_ids=np.array([d], np.int32), draft_probs=q,
              cu_num_draft=np.array([0, 1], np.int32), temperature=np.ones(1, np.float32),
              is_greedy=np.zeros(1, np.uint8), seed=11)
    o = oracle.run(b, u_override=np.array([u], np.float32))
    return int(o["num_sampled"][0]) == 2          # draft accepted (then the bonus is drawn)


CASES = [(2, 1, 0.75), (4, 1, 0.75), (3, 3, 0.7), (7, 3, 0.9), (7, 7, 0.3), (16, 5, 0.55),
         (1024, 3, 0.45), (1024, 1000, 0.001)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,n,q_d", CASES)
def test_probs_mode_accepts_at_equality_and_rejects_one_ulp_above(V, n, q_d, dtype):
    p_d = F32(1.0) / F32(n)                        # exp(0) / S with S = n
    ratio = p_d / F32(q_d)                          # binary32 quotient, correctly rounded
    assert ratio.dtype == np.float32
    assert _run(V, n, q_d, ratio, dtype)            # u == p/q: accepted (>=)
    assert not _run(V, n, q_d, np.nextafter(ratio, F32(np.inf)), dtype)
    assert _run(V, n, q_d, np.nextafter(ratio, F32(0)), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,n", [(2, 1), (2, 2), (3, 3), (8, 5), (1024, 7), (1024, 1024)])
def test_draft_ids_only_mode_accepts_at_equality_and_rejects_one_ulp_above(V, n, dtype):
    p_d = F32(1.0) / F32(n)                         # q(d) = 1 without draft probabilities
    assert _run(V, n, None, p_d, dtype)
    assert not _run(V, n, None, np.nextafter(p_d, F32(np.inf)), dtype)
    assert _run(V, n, None, np.nextafter(p_d, F32(0)), dtype)


def test_quotient_is_rounded_in_binary32():
    """Cases where fl(p / q) lies above the exact quotient: a comparison made in double would
    reject u = fl(p / q); the binary32 test accepts it."""
    hits = 0
    for V, n, q_d in CASES:
        p_d = F32(1.0) / F32(n)
        ratio = p_d / F32(q_d)
        if float(ratio) > float(p_d) / float(F32(q_d)):
            hits += 1
            assert _run(V, n, q_d, ratio)
    assert hits >= 3


def test_zero_target_probability_is_never_accepted():
    """A token outside the kept row (logit -inf) has p(d) = 0: rejected for every u in (0, 1),
    even the smallest uniform the generator can give, 2^-24."""
    assert not _run(4, 2, 0.5, F32(2.0 ** -24), d=3)
    assert not _run(4, 2, None, F32(2.0 ** -24), d=3)
