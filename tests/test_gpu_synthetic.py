"""GPU parity of synthetic acceptance ([spec-in-vllm] 7.2 / 7.4) and of the chunked-prefill
count correction ([MTP-eagle] get_num_sampled_and_rejected), against the oracle."""
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
    return workloads.make_batch(name=f"syn{seed}", data_seed=seed, verify_seed=seed * 31 + 5, K=Ks,
                                vocab_size=V, logits_dtype=dtype, sigma=2.0, zipf_coef=0.5,
                                q_mode=q_mode, q_noise=1.5, p_argmax=0.5,
                                temperature=rng.uniform(0.4, 1.4, n).astype(np.float32),
                                greedy=(rng.random(n) < greedy_frac).astype(np.uint8))


SYN = [
    # seed, V, K per request, dtype, q mode, rates
    (81, 1000, [3, 0, 5, 1, 2, 4, 0, 3] * 4, "f32", "none", [0.9, 0.7, 0.7, 0.4, 0.2]),
    (82, 30011, [4, 4, 2, 0, 3, 4, 1, 4], "bf16", "noisy", [0.8, 0.5, 0.3, 0.1]),   # q ignored
    (83, 20011, [5, 3, 0, 2, 5, 1], "bf16", "logits", [1.0, 1.0, 0.6]),             # K > rates
    (84, 7, [3, 1, 0, 2], "f32", "none", [0.5, 0.5, 0.5]),
]


@pytest.mark.parametrize("seed,V,Ks,dtype,q_mode,rates", SYN)
def test_synthetic_parity(seed, V, Ks, dtype, q_mode, rates):
    b = _batch(seed, V, Ks, dtype, q_mode)
    b.synthetic_rates = np.asarray(rates, np.float32)
    if b.num_draft_tokens > 2:
        b.draft_ids[1] = V                  # an invalid id is rejected in this mode too
    ref = oracle.run(b)
    assert_parity(b, gpu_run(b), ref)


def test_synthetic_target_length_and_switching_off():
    import speculative_decoding_verification_rejection_gb300 as sv

    b = _batch(85, 32000, [5] * 48, "bf16", "noisy", greedy_frac=0.1)
    ctx = sv.SpecVerify(b.num_reqs, 5, b.vocab_size, "bf16", True)
    try:
        ctx.set_synthetic_length(3.25)                  # 2 or 3 accepted drafts
        b.synthetic_rates = oracle.synthetic_rates(3.25, 5)
        got = gpu_run(b, ctx)                           # gpu_run sets the same rates again
        assert_parity(b, got, oracle.run(b))
        assert set(np.unique(got["num_sampled"] - 1)) <= {2, 3}
        b.synthetic_rates = None                        # off again: the ordinary test
        assert_parity(b, gpu_run(b, ctx), oracle.run(b))
        for bad in ([0.5, 0.7], [1.2], [-0.1], [float("nan")], [0.5] * (sv.SV_MAX_SYNTHETIC + 1)):
            with pytest.raises(sv.SpecVerifyError):
                ctx.set_synthetic(bad)
    finally:
        ctx.close()


@pytest.mark.parametrize("q_mode", ["noisy", "none", "logits"])
def test_partial_prefill_parity(q_mode):
    b = _batch(86, 12007, [3, 0, 4, 2, 5, 1, 0, 3, 2, 4], "bf16", q_mode)
    b.partial_prefill = np.zeros(b.num_reqs, np.uint8)
    b.partial_prefill[[0, 1, 6, 9]] = 1
    got = gpu_run(b)
    assert_parity(b, got, oracle.run(b))
    assert np.all(got["num_sampled"][[0, 1, 6, 9]] == 0)
    assert np.all(got["sampled"][[0, 1, 6, 9]] == -1)


def test_run_batch_equals_run():
    """spec_verify_run_batch with no extra fields gives spec_verify_run's outputs."""
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    b = workloads.workload(1)
    d = to_device(b)
    ctx = sv.SpecVerify(b.num_reqs, b.max_spec_len, b.vocab_size, "bf16", True)
    try:
        base = ctx.run(d["logits"], d["draft_ids"], d["draft_probs"], d["cu_num_draft"],
                       d["temperature"], d["is_greedy"], b.seed, row_stats=True)
        flags = torch.zeros(b.num_reqs, dtype=torch.uint8, device="cuda")
        other = ctx.run(d["logits"], d["draft_ids"], d["draft_probs"], d["cu_num_draft"],
                        d["temperature"], d["is_greedy"], b.seed, row_stats=True,
                        partial_prefill=flags)
        torch.cuda.synchronize()
        for x, y in zip(base, other):
            assert torch.equal(x, y)
    finally:
        ctx.close()
