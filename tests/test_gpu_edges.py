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


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,chunks", [(1001, 0), (1001, 512), (20011, 512), (20011, 0), (20011, 32768),
                                      (151936, 0)])
def test_tied_maxima_first_occurrence(dtype, V, chunks):
    """The row maximum planted several times per row: runs of consecutive copies (inside one
    64-byte pair and across the pairs of neighbouring lanes), copies far apart (other warps and,
    with small statistics chunks, other segments), at the first and the last element. The first
    occurrence is the argmax: in the row output and in what greedy requests emit."""
    Ks = [2, 3, 0, 4, 1, 2, 3, 1]
    b = _batch(208, V, Ks, dtype, "noisy", greedy_frac=0.5)
    rng = np.random.default_rng(208)
    x = np.minimum(rng.normal(0, 2, (b.num_rows, V)), 10.0).astype(np.float32)
    M = np.float32(16.0)
    for r in range(b.num_rows):
        kind = r % 5
        if kind == 0:      # a run: the same pair and the pairs after it
            j = int(rng.integers(0, V - 40))
            x[r, j:j + 40] = M
        elif kind == 1:    # two copies far apart
            j = int(rng.integers(0, V // 2))
            x[r, [j, j + V // 2]] = M
        elif kind == 2:    # the first element and elsewhere
            x[r, [0, int(rng.integers(1, V))]] = M
        elif kind == 3:    # the last element only
            x[r, V - 1] = M
        else:              # copies inside one 64-element line, then scattered
            j = int(rng.integers(0, V - 64)) & ~63
            x[r, [j + 37, j + 50, j + 63]] = M
            x[r, rng.integers(j + 64, V, 5) if j + 64 < V else []] = M
    b.logits = _as_dtype(x, dtype)
    got = gpu_run(b, chunks=chunks or None)
    assert_parity(b, got, oracle.run(b))
    first = np.argmax(x == M, axis=1)
    np.testing.assert_array_equal(got["row_argmax"], first)
