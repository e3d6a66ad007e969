"""GPU parity of the draft-logits input mode: q = softmax(draft_logits / T) computed inside the
call ([spec-in-vllm] 7.1 probabilistic drafting keeps the draft logits; 7.4 the statistics
kernel reduces target and draft logits), against the oracle on the same seeded batches."""
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


def _batch(seed, V, Ks, dtype, greedy_frac=0.25, temps=(0.3, 1.5), q_noise=1.5):
    rng = np.random.default_rng(seed)
    n = len(Ks)
    T = rng.uniform(*temps, n).astype(np.float32)
    g = (rng.random(n) < greedy_frac).astype(np.uint8)
    return workloads.make_batch(name=f"dl{seed}", data_seed=seed, verify_seed=seed * 104729 + 3,
                                K=Ks, vocab_size=V, logits_dtype=dtype, sigma=2.5, zipf_coef=0.5,
                                n_boost=3, boost=5.0, q_mode="logits", q_noise=q_noise,
                                temperature=T, greedy=g)


CASES = [
    # seed, V, K per request, dtype
    (21, 1000, [3, 0, 5, 1, 2, 4, 0, 3], "f32"),
    (22, 1001, [2, 2, 0, 6, 1], "bf16"),                 # odd V: unaligned draft rows
    (23, 7, [3, 1, 0, 2], "f32"),                        # tiny vocabulary
    (24, 129, [8, 0, 1], "bf16"),
    (25, 40000, [3, 2, 4, 0, 1, 5], "bf16"),             # several segments per row + ragged tail
    (26, 40003, [1, 3, 0, 2], "f32"),
    (27, 4004, [2, 4, 0, 3, 1], "bf16"),                 # bf16 rows 8-byte aligned
    (28, 65536, [0, 0, 0], "bf16"),                      # no drafts at all: bonus only
]


@pytest.mark.parametrize("seed,V,Ks,dtype", CASES)
def test_draft_logits_parity(seed, V, Ks, dtype):
    b = _batch(seed, V, Ks, dtype)
    b.temperature[0] = 0.0                  # T <= 0 means greedy
    if b.num_draft_tokens > 2:
        b.draft_ids[1] = V                  # out of range: rejected
        b.draft_ids[2] = -1
    assert_parity(b, gpu_run(b), oracle.run(b))


@pytest.mark.parametrize("q_noise", [0.05, 4.0])
def test_draft_logits_close_and_far_drafts(q_noise):
    """A draft close to the target (most drafts accepted, residual with few candidates) and a
    far one (early rejections, residual close to p)."""
    b = _batch(30 + int(q_noise * 10), 30011, [5] * 12, "bf16", greedy_frac=0.0, q_noise=q_noise)
    r = assert_parity(b, gpu_run(b), oracle.run(b))
    assert r["requests"] == 12


@pytest.mark.parametrize("c", [1, 3])
def test_workload_with_draft_logits(c):
    b = workloads.workload(c, draft_logits=True)
    got = gpu_run(b)
    r = assert_parity(b, got, oracle.run(b))
    assert got["error_word"] == 0
    print(f"{b.name}: {r['requests']} requests, {r['positions']} positions, ties {r['ties']}")


def test_same_tokens_as_probabilities_mode():
    """Giving the oracle's q = softmax(draft_logits / T) as draft_probs must reproduce the
    draft-logits run (counted ties aside: S_d is summed in another order)."""
    b = _batch(41, 20011, [4, 2, 5, 0, 3, 1, 4, 4], "bf16", greedy_frac=0.2)
    via_logits = gpu_run(b)
    q = oracle.draft_probs(b.draft_logits, True, b.cu_num_draft, b.temperature, b.is_greedy)
    b2 = workloads.Batch(**{**b.__dict__, "draft_probs": q, "draft_logits": None})
    via_probs = gpu_run(b2)
    same = [i for i in range(b.num_reqs)
            if np.array_equal(via_logits["sampled"][i], via_probs["sampled"][i])]
    assert len(same) >= b.num_reqs - 1
    assert_parity(b2, via_probs, oracle.run(b2))


@pytest.mark.parametrize("chunks", [2048, 8192, 65536])
def test_draft_logits_launch_shape_does_not_change_results(chunks):
    b = _batch(51, 30011, [3, 5, 0, 2, 4, 1, 3, 3], "bf16", greedy_frac=0.2)
    base = gpu_run(b)
    other = gpu_run(b, chunks=chunks)
    for k in ("sampled", "num_sampled", "num_rejected", "row_max", "row_argmax"):
        np.testing.assert_array_equal(other[k], base[k])
    np.testing.assert_allclose(other["row_sumexp"], base["row_sumexp"], rtol=1e-5)


def test_draft_logits_needs_the_mode_and_matching_inputs():
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    b = _batch(61, 1000, [2, 1], "f32")
    d = to_device(b)
    ctx = sv.SpecVerify(2, 2, 1000, "f32", False)
    try:
        with pytest.raises(sv.SpecVerifyError):           # context without the mode
            ctx.run(d["logits"], d["draft_ids"], None, d["cu_num_draft"], d["temperature"],
                    d["is_greedy"], 1, draft_logits=d["draft_logits"])
    finally:
        ctx.close()
    ctx = sv.SpecVerify(2, 2, 1000, "f32", True, draft_logits=True)
    try:
        with pytest.raises(ValueError):                    # both q inputs
            ctx.run(d["logits"], d["draft_ids"], torch.zeros(3, 1000, device="cuda:0"),
                    d["cu_num_draft"], d["temperature"], d["is_greedy"], 1,
                    draft_logits=d["draft_logits"])
        with pytest.raises(sv.SpecVerifyError):            # draft logits missing
            sv.spec_verify_run_draft_logits(ctx.ctx, d["logits"], d["draft_ids"], None,
                                            d["cu_num_draft"], d["temperature"], d["is_greedy"],
                                            1, 0, 2, 3, 2, torch.empty(2, 3, dtype=torch.int32,
                                                                       device="cuda:0"),
                                            torch.empty(2, dtype=torch.int32, device="cuda:0"),
                                            torch.empty(2, dtype=torch.int32, device="cuda:0"))
        out = ctx.run(d["logits"], d["draft_ids"], None, d["cu_num_draft"], d["temperature"],
                      d["is_greedy"], b.seed, draft_logits=d["draft_logits"], row_stats=True)
        torch.cuda.synchronize()
        ref = oracle.run(b)
        np.testing.assert_array_equal(out[1].cpu().numpy(), ref["num_sampled"])
    finally:
        ctx.close()


def test_draft_logits_graph_capture_and_replay():
    """The draft-logits call captured in a CUDA graph: a replay gives the direct call's results."""
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    b = _batch(71, 12007, [3, 4, 0, 2, 5, 1], "bf16", greedy_frac=0.2)
    d = to_device(b)
    ctx = sv.SpecVerify(b.num_reqs, 5, b.vocab_size, "bf16", False, draft_logits=True)
    outs = (torch.empty((b.num_reqs, 6), dtype=torch.int32, device="cuda"),
            torch.empty(b.num_reqs, dtype=torch.int32, device="cuda"),
            torch.empty(b.num_reqs, dtype=torch.int32, device="cuda"))

    def call():
        ctx.run(d["logits"], d["draft_ids"], None, d["cu_num_draft"], d["temperature"],
                d["is_greedy"], b.seed, max_spec_len=5, out=outs, draft_logits=d["draft_logits"])

    call()
    torch.cuda.synchronize()
    direct = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for o in outs:
        o.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    for a, c in zip(outs, direct):
        assert torch.equal(a, c)
    del g
    ctx.close()
