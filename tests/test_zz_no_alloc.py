"""The entry point that allocates nothing, against the regular context-based entry point.

Some callers cannot allocate device memory when they verify a batch: code that runs inside
another framework's memory pool or a plugin's execute call, where cudaMalloc is forbidden or
would synchronise the device, or processes that reserve all device memory up front. For them
spec_verify_run_noalloc keeps its scratch in a fixed static device array of the library.
Here it is called through the C ABI twice in a row, on batches of different shapes and
types (so anything left over in the shared array from the first call would show), and its
outputs must equal those of spec_verify_run on the same inputs.
"""
import numpy as np
import pytest

import oracle
import workloads
from _parity import S_RTOL, assert_parity, to_device

pytestmark = pytest.mark.gpu


def _context_run(batch):
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    ctx = sv.SpecVerify(batch.num_reqs, batch.max_spec_len, batch.vocab_size, batch.logits_dtype,
                        batch.draft_probs is not None)
    d = to_device(batch)
    outs = ctx.run(d["logits"], d["draft_ids"], d["draft_probs"], d["cu_num_draft"],
                   d["temperature"], d["is_greedy"], batch.seed, row_stats=True)
    torch.cuda.synchronize()
    res = [o.cpu().numpy() for o in outs]
    ctx.close()
    return res


def _noalloc_run(batch):
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    d = to_device(batch)
    n, nd, k = batch.num_reqs, batch.num_draft_tokens, batch.max_spec_len
    R = nd + n
    outs = [torch.full((n, k + 1), -7, dtype=torch.int32, device="cuda"),
            torch.full((n,), -7, dtype=torch.int32, device="cuda"),
            torch.full((n,), -7, dtype=torch.int32, device="cuda"),
            torch.zeros(R, dtype=torch.float32, device="cuda"),
            torch.zeros(R, dtype=torch.float32, device="cuda"),
            torch.zeros(R, dtype=torch.int32, device="cuda")]
    sv.spec_verify_run_noalloc(d["logits"], batch.logits_dtype, batch.vocab_size, d["draft_ids"],
                               d["draft_probs"], d["cu_num_draft"], d["temperature"],
                               d["is_greedy"], batch.seed, 0, n, nd, k, *outs)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs]


def _same(a, b):
    for k in (0, 1, 2, 3, 5):                       # tokens, lengths, row max, argmax: exact
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_allclose(a[4], b[4], rtol=S_RTOL)  # sum of exponentials


def test_noalloc_matches_context_entry_point_on_two_calls_in_a_row():
    import torch

    assert torch.cuda.is_available(), "this test needs a CUDA device"
    first = workloads.workload(1)                   # bf16, draft probs, greedy mix
    rng = np.random.default_rng(5)
    second = workloads.make_batch(                  # fp32, draft ids only, ragged vocabulary
        name="noalloc-2", data_seed=21, verify_seed=(3 << 33) + 21, K=[0, 4, 2, 5, 1, 3, 0, 2],
        vocab_size=50021, logits_dtype="f32", sigma=2.0, zipf_coef=1.1, q_mode="none",
        temperature=rng.uniform(0.4, 1.4, 8).astype(np.float32),
        greedy=np.array([0, 0, 1, 0, 0, 0, 1, 0], np.uint8))
    for batch in (first, second):
        _same(_noalloc_run(batch), _context_run(batch))


NAMES = ("sampled", "num_sampled", "num_rejected", "row_max", "row_sumexp", "row_argmax")


@pytest.mark.parametrize("c", [0, 1, 2, 3, 4])
def test_noalloc_matches_the_oracle_on_the_workloads(c):
    """Every workload at full size fits the static array; this entry point takes its race's
    line maxima from the raced rows themselves (it has no room to keep them), so it is checked
    against the oracle directly, by the parity rules of every other GPU test."""
    import speculative_decoding_verification_rejection_gb300 as sv

    b = workloads.workload(c)
    got = dict(zip(NAMES, _noalloc_run(b)))
    r = assert_parity(b, got, oracle.run(b))
    assert sv.spec_verify_noalloc_last_error() == 0
    print(f"workload {c}: {r['requests']} requests, ties {r['ties']}")


def test_noalloc_error_word_reports_an_inconsistent_batch_and_is_cleared():
    import speculative_decoding_verification_rejection_gb300 as sv

    b = workloads.workload(0)
    assert sv.spec_verify_noalloc_last_error() == 0
    bad = workloads.Batch(**{**b.__dict__})
    bad.cu_num_draft = np.array([0, 3, 2, 9, 12], np.int32)          # decreasing pair
    got = _noalloc_run(bad)
    assert np.all(got[1] == 0) and np.all(got[0] == -1)
    assert sv.spec_verify_noalloc_last_error() & sv.SV_ERR_BATCH
    assert sv.spec_verify_noalloc_last_error() == 0                  # read and cleared
    _same(_noalloc_run(b), _context_run(b))                          # the array is still fine


def test_noalloc_rejects_sizes_beyond_its_limits():
    import speculative_decoding_verification_rejection_gb300 as sv

    L = sv.lib()
    rc = L.spec_verify_run_noalloc(None, sv.SV_BF16, 262144 + 8, None, None, None, None, None, 0, 0,
                                   1, 0, 0, None, None, None, None, None, None, None)
    assert rc == sv.SV_ECAPACITY
    rc = L.spec_verify_run_noalloc(None, sv.SV_BF16, 1024, None, None, None, None, None, 0, 0,
                                   1025, 0, 0, None, None, None, None, None, None, None)
    assert rc == sv.SV_ECAPACITY
    rc = L.spec_verify_run_noalloc(None, sv.SV_F32, 1024, None, None, None, None, None, 0, 0,
                                   1000, 8000, 8, None, None, None, None, None, None, None)
    assert rc == sv.SV_ECAPACITY                    # 9000 rows > 8192
