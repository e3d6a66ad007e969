"""GPU parity at the edges: a vocabulary of one token, masked (-inf) and huge logits, flat rows
(every key ties but the clocks), long drafts, many small requests, a large vocabulary and extreme
temperatures, each against the oracle."""
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


def _batch(seed, V, Ks, dtype, q_mode, greedy_frac=0.2, temps=(0.5, 1.5)):
    rng = np.random.default_rng(seed)
    n = len(Ks)
    return workloads.make_batch(name=f"edge{seed}", data_seed=seed, verify_seed=seed * 11 + 3, K=Ks,
                                vocab_size=V, logits_dtype=dtype, sigma=2.0, zipf_coef=0.5,
                                q_mode=q_mode, q_noise=1.0, p_argmax=0.5,
                                temperature=rng.uniform(*temps, n).astype(np.float32),
                                greedy=(rng.random(n) < greedy_frac).astype(np.uint8))


def _as_dtype(x, dtype):
    x = np.asarray(x, np.float32)
    if dtype == "bf16":
        return (x.view(np.uint32) >> 16).astype(np.uint16)   # exact for the values used here
    return x


@pytest.mark.parametrize("dtype,q_mode", [("f32", "none"), ("bf16", "noisy"), ("f32", "noisy")])
def test_vocabulary_of_one(dtype, q_mode):
    """Every draft is token 0: accepted (p = q = 1), or, without q, the only token is both the
    draft and the whole residual: the draw falls back to p."""
    b = _batch(201, 1, [3, 0, 2, 1, 4], dtype, q_mode)
    assert_parity(b, gpu_run(b), oracle.run(b))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_masked_and_huge_logits(dtype):
    b = _batch(202, 3000, [3, 2, 0, 4, 1, 3], dtype, "none")
    rng = np.random.default_rng(202)
    x = rng.normal(0, 2, (b.num_rows, 3000)).astype(np.float32)
    x[:, rng.random(3000) < 0.7] = -np.inf        # a masked vocabulary: 70 % of tokens
    x[1, 5] = 1.0e4                               # one dominant token
    x[3, 7] = x[3, 9] = 3.0e3                     # two tied dominant tokens
    x[:, 11] = np.maximum(x[:, 11], -50.0)        # keep token 11 live
    b.logits = _as_dtype(x, dtype)
    assert_parity(b, gpu_run(b), oracle.run(b))


def test_flat_rows_tie_everywhere():
    """All logits equal: the argmax is token 0, the race is decided by the clocks alone."""
    b = _batch(203, 5000, [2, 3, 1, 0], "bf16", "none", greedy_frac=0.5)
    b.logits = np.full((b.num_rows, 5000), _as_dtype(np.float32(0.25), "bf16"), np.uint16)
    got = gpu_run(b)
    assert_parity(b, got, oracle.run(b))
    assert np.all(got["row_argmax"] == 0)


def test_long_drafts():
    b = _batch(204, 5000, [24, 0, 17, 9, 24, 3, 1, 12], "bf16", "noisy", greedy_frac=0.25)
    assert_parity(b, gpu_run(b), oracle.run(b))


def test_many_small_requests():
    rng = np.random.default_rng(205)
    Ks = rng.integers(0, 5, 2048)
    b = _batch(205, 1000, list(Ks), "f32", "noisy", greedy_frac=0.3)
    r = assert_parity(b, gpu_run(b), oracle.run(b))
    assert r["requests"] == 2048


def test_large_vocabulary():
    b = _batch(206, 262144, [3, 0, 2, 1], "bf16", "noisy", greedy_frac=0.0)
    assert_parity(b, gpu_run(b), oracle.run(b))


@pytest.mark.parametrize("T", [1e-4, 1e-2, 50.0, 1e4])
def test_extreme_temperatures(T):
    b = _batch(207, 20011, [3, 2, 4, 0, 1, 3], "bf16", "noisy", greedy_frac=0.0, temps=(T, T))
    assert_parity(b, gpu_run(b), oracle.run(b))
