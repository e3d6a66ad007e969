"""GPU parity of the fp64 Gumbel option ([spec-in-vllm] 7.3: use_fp64_gumbel, the race noise
drawn in double precision) against the oracle's binary64 races: the five workloads at full
size, then the option combined with the other per-call inputs."""
import numpy as np
import pytest

import oracle
import workloads
from _parity import assert_parity, gpu_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    import torch

    assert torch.cuda.is_available(), "these tests need a CUDA device"
    import speculative_decoding_verification_rejection_gb300 as sv

    sv.lib()


@pytest.mark.parametrize("c", [0, 1, 2, 3, 4])
def test_fp64_workload_parity(c):
    b = workloads.workload(c)
    b.fp64_gumbel = True
    got = gpu_run(b)
    r = assert_parity(b, got, oracle.run(b))
    assert got["error_word"] == 0
    print(f"workload {c} fp64: {r['requests']} requests, ties {r['ties']}")


def _batch(seed, V, Ks, dtype, q_mode, greedy_frac=0.2):
    rng = np.random.default_rng(seed)
    n = len(Ks)
    return workloads.make_batch(name=f"f64_{seed}", data_seed=seed, verify_seed=seed * 31 + 7,
                                K=Ks, vocab_size=V, logits_dtype=dtype, sigma=2.0, zipf_coef=0.8,
                                n_boost=3, boost=5.0, q_mode=q_mode, q_noise=1.5, p_argmax=0.6,
                                temperature=rng.uniform(0.3, 1.5, n).astype(np.float32),
                                greedy=(rng.random(n) < greedy_frac).astype(np.uint8))


CASES = [
    # seed, V, K per request, dtype, q mode
    (201, 1000, [3, 0, 5, 1, 2, 4, 0, 3] * 2, "f32", "noisy"),
    (202, 1001, [2, 2, 0, 6, 1] * 2, "bf16", "none"),
    (203, 40000, [3, 2, 4, 0, 1, 5], "bf16", "indep"),
    (204, 4004, [2, 4, 0, 3, 1], "bf16", "logits"),       # draft logits: q computed in the call
    (205, 7, [3, 1, 0, 2] * 4, "f32", "noisy"),            # tiny vocabulary
    (206, 65536, [2, 5, 3, 0, 1, 4, 2, 3], "f32", "none"),
]


@pytest.mark.parametrize("seed,V,Ks,dtype,q_mode", CASES)
def test_fp64_custom_parity(seed, V, Ks, dtype, q_mode):
    b = _batch(seed, V, Ks, dtype, q_mode)
    b.fp64_gumbel = True
    assert_parity(b, gpu_run(b), oracle.run(b))


def test_fp64_with_processors_and_synthetic():
    b = _batch(207, 30011, [4, 4, 2, 0, 3, 4, 1, 4] * 2, "bf16", "noisy")
    workloads.add_penalty(b, 207, history=(50, 200))
    rng = np.random.default_rng(208)
    b.top_k = rng.choice(np.array([0, 30, 300], np.int32), b.num_reqs).astype(np.int32)
    b.top_p = rng.choice(np.array([0.85, 1.0], np.float32), b.num_reqs).astype(np.float32)
    b.fp64_gumbel = True
    assert_parity(b, gpu_run(b), oracle.run(b))
    b.synthetic_rates = np.array([0.9, 0.6, 0.5, 0.2], np.float32)
    assert_parity(b, gpu_run(b), oracle.run(b))


def test_fp64_option_changes_only_the_races_on_the_gpu():
    b = workloads.workload(1)
    g32 = gpu_run(b)
    b.fp64_gumbel = True
    g64 = gpu_run(b)
    for k in ("num_sampled", "num_rejected", "row_max", "row_argmax"):
        np.testing.assert_array_equal(g64[k], g32[k])
    greedy = (b.is_greedy != 0) | ~(b.temperature > 0)
    np.testing.assert_array_equal(g64["sampled"][greedy], g32["sampled"][greedy])
    assert (g64["sampled"] != g32["sampled"]).any(axis=1)[~greedy].mean() > 0.5
