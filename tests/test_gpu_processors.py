"""GPU parity of the logits processors against the oracle: the frequency penalty ([MTP-eagle]
其他 / 重复惩罚), applied in the statistics pass and wherever the verifier reads a logit, and
the sampling constraints top-k / top-p ([spec-notes] 8.2; [mini-sglang])."""
import numpy as np
import pytest

import oracle
import workloads
from _parity import assert_parity, gpu_run, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    import torch

    assert torch.cuda.is_available(), "these tests need a CUDA device"
    import speculative_decoding_verification_rejection_gb300 as sv

    sv.lib()


def _batch(seed, V, Ks, dtype, q_mode, greedy_frac=0.25):
    rng = np.random.default_rng(seed)
    n = len(Ks)
    return workloads.make_batch(name=f"proc{seed}", data_seed=seed, verify_seed=seed * 7 + 1, K=Ks,
                                vocab_size=V, logits_dtype=dtype, sigma=2.0, zipf_coef=0.7,
                                n_boost=4, boost=4.0, q_mode=q_mode, q_noise=1.2, p_argmax=0.6,
                                temperature=rng.uniform(0.4, 1.4, n).astype(np.float32),
                                greedy=(rng.random(n) < greedy_frac).astype(np.uint8))


PEN = [
    # seed, V, K per request, dtype, q mode
    (91, 1000, [3, 0, 5, 1, 2, 4, 0, 3], "f32", "noisy"),
    (92, 1001, [2, 2, 0, 6, 1], "bf16", "none"),            # odd V: unaligned counts rows
    (93, 40000, [3, 2, 4, 0, 1, 5], "bf16", "noisy"),       # several segments per row
    (94, 40003, [1, 3, 0, 2], "f32", "indep"),
    (95, 4004, [2, 4, 0, 3, 1], "bf16", "logits"),
    (96, 7, [3, 1, 0, 2], "f32", "noisy"),                 # tiny vocabulary
    (97, 129, [8, 0, 1], "bf16", "none"),
]


@pytest.mark.parametrize("seed,V,Ks,dtype,q_mode", PEN)
def test_frequency_penalty_parity(seed, V, Ks, dtype, q_mode):
    b = _batch(seed, V, Ks, dtype, q_mode)
    workloads.add_penalty(b, seed, history=(5, 60), top_n=min(V, 20), extra_rows=3,
                          shuffle_rows=seed % 2 == 1)
    if b.num_draft_tokens > 2:                  # a repeated draft: counted at later positions
        b.draft_ids[1] = b.draft_ids[0]
    got = gpu_run(b)
    assert_parity(b, got, oracle.run(b))
    assert got["error_word"] == 0


def test_frequency_penalty_workload_style():
    b = workloads.workload(1)
    workloads.add_penalty(b, 5)
    assert_parity(b, gpu_run(b), oracle.run(b))


@pytest.mark.parametrize("chunks", [2048, 8192, 65536])
def test_penalty_launch_shape_does_not_change_results(chunks):
    b = _batch(98, 30011, [3, 5, 0, 2, 4, 1, 3, 3], "bf16", "noisy", greedy_frac=0.2)
    workloads.add_penalty(b, 98, history=(100, 400))
    base = gpu_run(b)
    other = gpu_run(b, chunks=chunks)
    for k in ("sampled", "num_sampled", "num_rejected", "row_max", "row_argmax"):
        np.testing.assert_array_equal(other[k], base[k])
    np.testing.assert_allclose(other["row_sumexp"], base["row_sumexp"], rtol=1e-5)


def test_bad_counts_row_is_reported_and_skips_the_penalty():
    b = _batch(99, 2000, [2, 3, 1, 0], "f32", "noisy")
    workloads.add_penalty(b, 99, history=(50, 100), top_n=10)
    b.counts_row = np.array([0, 1, 7, 3], np.int32)      # 7 is outside the 4 count rows
    got = gpu_run(b)
    assert_parity(b, got, oracle.run(b))
    import speculative_decoding_verification_rejection_gb300 as sv
    assert got["error_word"] & sv.SV_ERR_COUNTS


def test_malformed_cu_num_draft_with_penalty_and_constraints():
    """The statistics and selection kernels read cu_num_draft before the verify kernel has
    checked it; with a penalty they take each position's earlier drafts from it. A malformed
    prefix sum (an entry far below 0, one far above the number of drafts, a decreasing pair)
    must only produce empty rows and SV_ERR_BATCH, and leave the context usable."""
    import speculative_decoding_verification_rejection_gb300 as sv

    b = _constrain(_batch(111, 3001, [2, 3, 1, 0, 4], "bf16", "noisy"), 111, [0, 40], [0.9, 1.0])
    workloads.add_penalty(b, 111, history=(20, 80), top_n=20)
    nd = b.num_draft_tokens
    ctx = sv.SpecVerify(8, 6, 3001, "bf16", True)
    try:
        for cu in ([0, -1000000, 5, 6, 6, nd], [0, 2, 1 << 30, 6, 6, nd], [0, 2, 5, 4, 6, nd],
                   [0, 2, 5, 6, 6, nd + 7], [7, 2, 5, 6, 6, nd]):
            bad = workloads.Batch(**{**b.__dict__})
            bad.cu_num_draft = np.array(cu, np.int32)
            got = gpu_run(bad, ctx, max_spec_len=6)
            assert got["error_word"] & sv.SV_ERR_BATCH, cu
            assert np.all(got["num_sampled"] == 0) and np.all(got["sampled"] == -1), cu
        ok = gpu_run(b, ctx, max_spec_len=6)
        assert ok["error_word"] == 0
        assert_parity(b, ok, oracle.run(b, max_spec_len=6))
    finally:
        ctx.close()


def test_penalty_arguments_must_come_together():
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    b = _batch(100, 1000, [2, 1], "f32", "noisy")
    d = to_device(b)
    ctx = sv.SpecVerify(2, 2, 1000, "f32", True)
    try:
        with pytest.raises(sv.SpecVerifyError):
            ctx.run(d["logits"], d["draft_ids"], d["draft_probs"], d["cu_num_draft"],
                    d["temperature"], d["is_greedy"], 1,
                    frequency_penalty=torch.ones(2, device="cuda"))
    finally:
        ctx.close()


def _constrain(b, seed, k_choices, p_choices):
    rng = np.random.default_rng([seed, 77])
    b.top_k = rng.choice(np.asarray(k_choices, np.int32), b.num_reqs).astype(np.int32)
    b.top_p = rng.choice(np.asarray(p_choices, np.float32), b.num_reqs).astype(np.float32)
    return b


SEL = [
    # seed, V, K per request, dtype, q mode, top_k choices, top_p choices
    (101, 1000, [3, 0, 5, 1, 2, 4, 0, 3] * 3, "f32", "noisy", [0, 1, 5, 50, 999], [1.0, 0.9, 0.5]),
    (102, 1001, [2, 2, 0, 6, 1] * 3, "bf16", "none", [0, 20], [1.0, 0.95, 1e-9]),
    (103, 40000, [3, 2, 4, 0, 1, 5], "bf16", "noisy", [0, 40, 4000], [0.8, 0.99]),
    (104, 40003, [1, 3, 0, 2] * 2, "f32", "indep", [0, 7], [0.7, 1.0]),
    (105, 4004, [2, 4, 0, 3, 1], "bf16", "logits", [0, 100], [0.9]),
    (106, 7, [3, 1, 0, 2] * 3, "f32", "noisy", [0, 2, 3, 6, 7], [1.0, 0.6]),
    (107, 129, [8, 0, 1] * 3, "bf16", "none", [0, 64], [0.3, 1.0]),
]


@pytest.mark.parametrize("seed,V,Ks,dtype,q_mode,ks,ps", SEL)
def test_top_k_top_p_parity(seed, V, Ks, dtype, q_mode, ks, ps):
    b = _constrain(_batch(seed, V, Ks, dtype, q_mode), seed, ks, ps)
    got = gpu_run(b)
    r = assert_parity(b, got, oracle.run(b))
    assert got["error_word"] == 0
    print(f"{seed}: ties {r['ties']}")


def test_constraints_with_penalty_and_synthetic():
    b = _constrain(_batch(108, 30011, [4, 4, 2, 0, 3, 4, 1, 4] * 2, "bf16", "noisy"), 108,
                   [0, 30, 300], [0.85, 1.0])
    workloads.add_penalty(b, 108, history=(100, 300))
    assert_parity(b, gpu_run(b), oracle.run(b))
    b.synthetic_rates = np.array([0.9, 0.5, 0.5, 0.2], np.float32)
    assert_parity(b, gpu_run(b), oracle.run(b))


def test_selection_beyond_the_shared_pool():
    """Flat rows (every logit within 1/8 nat: the first bin holds the whole row) and rows of
    few distinct values (a boundary group larger than the in-memory pool)."""
    V = 20000
    b = _batch(109, V, [2, 1, 3, 0], "f32", "none", greedy_frac=0.0)
    rng = np.random.default_rng(109)
    flat = rng.uniform(0.0, 0.1, (b.num_rows, V)).astype(np.float32)
    flat[2] = np.repeat(np.array([1.0, 0.5, 0.25, 0.0], np.float32), V // 4)   # 4 values
    flat[5] = np.float32(0.0)                                                # one value
    b.logits = flat
    b.temperature[:] = 1.0
    b.top_k = np.array([15000, 0, 4000, 9000], np.int32)
    b.top_p = np.array([1.0, 0.5, 0.6, 0.97], np.float32)
    assert_parity(b, gpu_run(b), oracle.run(b))


def test_constrained_workload_style():
    b = workloads.workload(3, num_reqs=48)
    b.top_p = np.full(b.num_reqs, 0.9, np.float32)
    b.top_k = np.where(np.arange(b.num_reqs) % 2 == 0, 0, 50).astype(np.int32)
    got = gpu_run(b)
    r = assert_parity(b, got, oracle.run(b))
    print(f"workload 3 (48 requests) with top-p 0.9 / top-k 50: ties {r['ties']}")


@pytest.mark.parametrize("dtype,V", [("bf16", 5000), ("f32", 3001)])
def test_penalty_long_drafts_and_extreme_counts(dtype, V):
    """More than 32 earlier drafts (the statistics and selection passes then add them in every
    round), counts of 2^23 and beyond (converted by the exact fallback) and negative counts,
    with and without top-k / top-p."""
    b = _batch(110, V, [40, 3, 0, 35, 2], dtype, "noisy", greedy_frac=0.0)
    workloads.add_penalty(b, 110, history=(20, 80), top_n=20)
    rng = np.random.default_rng([110, V])
    cols = rng.choice(V, 8, replace=False)
    b.output_bin_counts[0, cols[:4]] = [1 << 23, (1 << 24) + 1, (1 << 30) + 3, -3]
    b.output_bin_counts[3, cols[4:]] = [(1 << 23) + 5, -1, 7, (1 << 25) - 1]
    b.draft_ids[5:12] = b.draft_ids[0]          # repeated drafts: counted at later positions
    b.draft_ids[45:50] = b.draft_ids[44]
    assert_parity(b, gpu_run(b), oracle.run(b))
    _constrain(b, 110, [0, 30], [0.9, 1.0])
    assert_parity(b, gpu_run(b), oracle.run(b))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_constraints_on_masked_and_huge_logits(dtype):
    """top-k / top-p over rows with a masked vocabulary (-inf on 70 % of tokens) and dominant
    tokens: most 64-token groups lie below the threshold and are left out of the race."""
    V = 3000
    b = _batch(111, V, [3, 2, 0, 4, 1, 3], dtype, "none")
    rng = np.random.default_rng(111)
    x = rng.normal(0, 2, (b.num_rows, V)).astype(np.float32)
    x[:, rng.random(V) < 0.7] = -np.inf
    x[1, 5] = 1.0e4
    x[3, 7] = x[3, 9] = 3.0e3
    x[:, 11] = np.maximum(x[:, 11], -50.0)
    b.logits = x if dtype == "f32" else (x.view(np.uint32) >> 16).astype(np.uint16)  # truncated
    _constrain(b, 111, [0, 1, 3, 40], [0.5, 0.95, 1.0])
    assert_parity(b, gpu_run(b), oracle.run(b))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [4096, 4099])
def test_penalised_maxima_next_to_raw_ones(dtype, V):
    """Penalised rows whose maximum is tied between a counted token (its value changed by the
    penalty) and a raw one close by, in either order, at the row's first and last token, and
    made by an earlier draft: the first occurrence of the processed maximum must come back as
    the argmax (greedy requests emit it) and the statistics must match the oracle."""
    Ks = [3, 2, 4, 1, 0, 2]
    b = _batch(98, V, Ks, dtype, "noisy", greedy_frac=1.0)
    n, R = b.num_reqs, b.num_rows
    rng = np.random.default_rng(98)
    x = np.minimum(rng.normal(0, 1.5, (R, V)), 4.0).astype(np.float32)
    counts = np.zeros((n, V), np.int32)
    f = np.full(n, -2.0, np.float32)           # a boost: y = l + 2 n
    cu = b.cu_num_draft
    rows = lambda i: range(int(cu[i]) + i, int(cu[i + 1]) + i + 1)  # noqa: E731
    for r in rows(0):                          # counted token first, raw tie after it
        x[r, 100], x[r, 105] = 6.0, 8.0
    counts[0, 100] = 1
    for r in rows(1):                          # raw token first, counted tie after it
        x[r, 70], x[r, 80] = 8.0, 6.0
    counts[1, 80] = 1
    for r in rows(2):                          # the first token counted, a raw tie next to it
        x[r, 0], x[r, 3] = 6.0, 8.0
    counts[2, 0] = 1
    for r in rows(3):                          # the last token counted: the top
        x[r, V - 1] = 7.0
    counts[3, V - 1] = 1
    f[4] = 1.5                                 # a plain penalty on the top raw token
    for r in rows(4):
        x[r, 9] = 9.0
    counts[4, 9] = 2
    d = int(cu[5])                             # an earlier draft at position 1 lifts a token
    b.draft_ids[d] = 2000
    for r in rows(5):
        x[r, 2000], x[r, 2001] = 6.0, 8.0
    counts[5, 2000] = 0                        # only the draft counts it, from position 1 on
    b.logits = (x.view(np.uint32) >> 16).astype(np.uint16) if dtype == "bf16" else x
    b.output_bin_counts, b.counts_row, b.frequency_penalty = counts, None, f
    got = gpu_run(b)
    ref = oracle.run(b)
    assert_parity(b, got, ref)
    np.testing.assert_array_equal(got["row_argmax"], ref["row_argmax"])
    assert got["error_word"] == 0
