"""GPU: vocabulary-sharded verification through the C ABI. The ranks are emulated on one GPU as
independent launches (none waits on another); the exchange is a concatenation in rank order.
The sharded step must reproduce the oracle's unsharded step, and each rank's records the
oracle's side of the protocol."""
import numpy as np
import pytest

import oracle
import workloads
from _parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    import torch

    assert torch.cuda.is_available(), "these tests need a CUDA device"
    import speculative_decoding_verification_rejection_gb300 as sv

    sv.lib()


def _run_sharded(b, world):
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv
    from speculative_decoding_verification_rejection_gb300.shard import (ShardBackend, sharded_verify,
                                                                         vocab_bounds)
    dev = "cuda:0"
    bounds = [(lo, hi) for lo, hi in vocab_bounds(b.vocab_size, world) if hi > lo]
    logits = np.ascontiguousarray(b.logits)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).to(dev)  # noqa: E731
    ids, cu = t(b.draft_ids, np.int32), t(b.cu_num_draft, np.int32)
    T, g = t(b.temperature, np.float32), t(b.is_greedy, np.uint8)
    sides, ctxs = [], []
    for lo, hi in bounds:
        sl = np.ascontiguousarray(logits[:, lo:hi])
        lt = torch.from_numpy(sl.view(np.int16) if sl.dtype == np.uint16 else sl).to(dev)
        q = None if b.draft_probs is None else t(np.asarray(b.draft_probs)[:, lo:hi], np.float32)
        ctx = sv.SpecVerify(b.num_reqs, max(b.max_spec_len, 0), hi - lo, b.logits_dtype,
                            b.draft_probs is not None)
        ctxs.append(ctx)
        sides.append(ShardBackend(ctx, lo, b.vocab_size, lt, ids, q, cu, T, g, b.seed,
                                  max_spec_len=b.max_spec_len))
    w = len(sides)
    stats = [s.stats() for s in sides]
    all_stats = torch.cat(stats)
    races = [s.race(all_stats, w) for s in sides]
    all_races = torch.cat(races)
    outs = [s.finish(all_races, w, b.max_spec_len) for s in sides]
    torch.cuda.synchronize()
    res = [tuple(x.cpu().numpy() for x in o) for o in outs]
    recs = [x.cpu().numpy() for x in stats]
    for c in ctxs:
        c.close()
    # every rank emits the same rows
    for r in res[1:]:
        for a, c in zip(r, res[0]):
            np.testing.assert_array_equal(a, c)
    return res[0], bounds, recs


@pytest.mark.parametrize("c,world", [(0, 2), (1, 2), (1, 4), (2, 3), (4, 2), (3, 2)])
def test_sharded_step_matches_the_unsharded_oracle(c, world):
    b = workloads.workload(c, num_reqs=48 if c == 3 else None)
    (sampled, ns, nr), _, _ = _run_sharded(b, world)
    ref = oracle.run(b)
    got = dict(sampled=sampled, num_sampled=ns, num_rejected=nr, row_max=ref["row_max"],
               row_sumexp=ref["row_sumexp"], row_argmax=ref["row_argmax"])
    assert_parity(b, got, ref)


def test_shard_records_match_the_oracle_side():
    b = workloads.workload(1)
    _, bounds, recs = _run_sharded(b, 2)
    for (lo, hi), rec in zip(bounds, recs):
        want = oracle.ShardOracle(b, lo, hi - lo).stats()
        got = rec.view(np.dtype([("max_logit", "<f4"), ("sumexp", "<f4"), ("argmax", "<i4"),
                                 ("draft_logit", "<f4"), ("draft_prob", "<f4"), ("r", "<i4")]))
        np.testing.assert_array_equal(got["max_logit"], want["ymax"])
        np.testing.assert_array_equal(got["argmax"], want["amax"])
        np.testing.assert_array_equal(np.isnan(got["draft_logit"]), np.isnan(want["ld"]))
        held = ~np.isnan(want["ld"])
        np.testing.assert_array_equal(got["draft_logit"][held], want["ld"][held])
        np.testing.assert_array_equal(got["draft_prob"][held], want["qd"][held])
        np.testing.assert_allclose(got["sumexp"], want["s"], rtol=1e-5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_shard_records_keep_the_first_of_tied_maxima(dtype):
    """Each row's maximum planted as runs and scattered copies, some in both shards: every rank's
    record holds the first occurrence in its own slice, and the step the lowest overall."""
    V = 8192 + 64 * 5
    rng = np.random.default_rng(209)
    Ks = [2, 3, 1, 0, 2]
    b = workloads.make_batch(name="shard-ties", data_seed=209, verify_seed=210, K=Ks, vocab_size=V,
                             logits_dtype=dtype, sigma=2.0, q_mode="noisy", q_noise=1.0,
                             temperature=rng.uniform(0.5, 1.5, len(Ks)).astype(np.float32),
                             greedy=np.array([1, 0, 1, 1, 0], np.uint8))
    x = np.minimum(rng.normal(0, 2, (b.num_rows, V)), 10.0).astype(np.float32)
    for r in range(b.num_rows):
        j = int(rng.integers(0, V - 40))
        x[r, j:j + 1 + r % 40] = 16.0
        x[r, rng.integers(0, V, 4)] = 16.0
    b.logits = (x.view(np.uint32) >> 16).astype(np.uint16) if dtype == "bf16" else x
    vals = (b.logits.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else x
    (sampled, ns, nr), bounds, recs = _run_sharded(b, 2)
    for (lo, hi), rec in zip(bounds, recs):
        got = rec.view(np.dtype([("max_logit", "<f4"), ("sumexp", "<f4"), ("argmax", "<i4"),
                                 ("draft_logit", "<f4"), ("draft_prob", "<f4"), ("r", "<i4")]))
        xs = vals[:, lo:hi]
        first = lo + np.argmax(xs == xs.max(axis=1, keepdims=True), axis=1)
        np.testing.assert_array_equal(got["argmax"], first)
    ref = oracle.run(b)
    assert_parity(b, dict(sampled=sampled, num_sampled=ns, num_rejected=nr, row_max=ref["row_max"],
                          row_sumexp=ref["row_sumexp"], row_argmax=ref["row_argmax"]), ref)


def test_misaligned_shard_is_refused():
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    ctx = sv.SpecVerify(2, 2, 500, "f32", False)
    try:
        lg = torch.zeros((4, 500), device="cuda")
        ids = torch.zeros(2, dtype=torch.int32, device="cuda")
        cu = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
        T = torch.ones(2, device="cuda")
        g = torch.zeros(2, dtype=torch.uint8, device="cuda")
        out = torch.empty(4 * sv.SHARD_RECORD_BYTES, dtype=torch.uint8, device="cuda")
        with pytest.raises(sv.SpecVerifyError):
            sv.spec_verify_shard_stats(ctx.ctx, lg, 100, ids, None, cu, T, g, 2, 2, 2, out)
    finally:
        ctx.close()
