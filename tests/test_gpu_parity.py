"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by element."""
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


@pytest.mark.parametrize("c", [0, 1, 2, 3, 4])
def test_workload_parity(c):
    b = workloads.workload(c)
    ref = oracle.run(b)
    got = gpu_run(b)
    r = assert_parity(b, got, ref)
    assert got["error_word"] == 0
    print(f"workload {c}: {r['requests']} requests, {r['positions']} positions, ties {r['ties']}, "
          f"max S rel err {r['max_sumexp_rel']:.2e}")


def _custom(seed, V, Ks, dtype, q_mode, greedy_frac=0.25, temps=(0.3, 1.5), sigma=2.5, zipf=0.0):
    rng = np.random.default_rng(seed)
    n = len(Ks)
    T = rng.uniform(*temps, n).astype(np.float32)
    g = (rng.random(n) < greedy_frac).astype(np.uint8)
    return workloads.make_batch(name=f"custom{seed}", data_seed=seed, verify_seed=seed * 7919 + (1 << 40),
                                K=Ks, vocab_size=V, logits_dtype=dtype, sigma=sigma, zipf_coef=zipf,
                                n_boost=3, boost=5.0, q_mode=q_mode, q_noise=1.5, temperature=T,
                                greedy=g)


CUSTOM = [
    # seed, V, K per request, dtype, q mode
    (1, 1000, [3, 0, 5, 1, 2, 4, 0, 3], "f32", "noisy"),
    (2, 1001, [2, 2, 0, 6, 1], "bf16", "noisy"),            # odd V: unaligned rows
    (3, 5003, [4, 1, 0, 3, 2, 5, 2, 1, 0, 4], "bf16", "none"),
    (4, 40000, [3, 2, 4, 0, 1, 5], "bf16", "noisy"),       # several splits per row + ragged tail
    (5, 40003, [1, 3, 0, 2], "f32", "none"),
    (6, 65536, [2, 5, 3, 0, 1, 4, 2, 3], "f32", "indep"),
    (7, 7, [3, 1, 0, 2], "f32", "noisy"),                  # tiny vocabulary
    (8, 129, [8, 0, 1], "bf16", "indep"),
    (9, 4004, [2, 4, 0, 3, 1], "bf16", "noisy"),          # V % 8 == 4: bf16 rows 8-byte aligned
    (10, 2052, [5, 5, 5, 5, 5, 5, 5, 5], "f32", "noisy"),  # rows a little above the minimum chunk
]


@pytest.mark.parametrize("seed,V,Ks,dtype,q_mode", CUSTOM)
def test_custom_parity(seed, V, Ks, dtype, q_mode):
    b = _custom(seed, V, Ks, dtype, q_mode)
    b.temperature[0] = 0.0                  # T <= 0 means greedy
    if b.num_draft_tokens > 2:
        b.draft_ids[1] = V                  # out of range: rejected
        b.draft_ids[2] = -1
    ref = oracle.run(b)
    got = gpu_run(b)
    assert_parity(b, got, ref)


@pytest.mark.parametrize("chunks", [2048, 4096, 65536])
def test_launch_shape_does_not_change_results(chunks):
    b = _custom(11, 30011, [3, 5, 0, 2, 4, 1, 3, 3], "bf16", "noisy", greedy_frac=0.2)
    base = gpu_run(b)
    other = gpu_run(b, chunks=chunks)
    for k in ("sampled", "num_sampled", "num_rejected", "row_max", "row_argmax", "row_sumexp"):
        if k == "row_sumexp":
            np.testing.assert_allclose(other[k], base[k], rtol=1e-5)
        else:
            np.testing.assert_array_equal(other[k], base[k])


def test_request_index_base_and_sharding():
    b = _custom(12, 20000, [3, 1, 4, 0, 2, 5, 3, 2, 1, 0], "bf16", "noisy", greedy_frac=0.0)
    full = gpu_run(b, max_spec_len=5)
    ref = oracle.run(b, max_spec_len=5)
    assert_parity(b, full, ref)
    cu = b.cu_num_draft
    cut = 4
    from workloads import Batch
    parts = []
    for lo, hi in ((0, cut), (cut, b.num_reqs)):
        r0, r1 = cu[lo] + lo, cu[hi] + hi
        sub = Batch(name="part", logits=b.logits[r0:r1], logits_dtype=b.logits_dtype,
                    vocab_size=b.vocab_size, draft_ids=b.draft_ids[cu[lo]:cu[hi]],
                    draft_probs=b.draft_probs[cu[lo]:cu[hi]],
                    cu_num_draft=(cu[lo:hi + 1] - cu[lo]).astype(np.int32),
                    temperature=b.temperature[lo:hi], is_greedy=b.is_greedy[lo:hi], seed=b.seed)
        parts.append(gpu_run(sub, max_spec_len=5, req_index_base=lo))
    np.testing.assert_array_equal(np.concatenate([p["sampled"] for p in parts]), full["sampled"])


def test_empty_residual_falls_back_to_p():
    """q = 2p leaves no positive residual: the token at a rejection is a draw from p."""
    V, n = 3000, 64
    b = _custom(13, V, [1] * n, "f32", "noisy", greedy_frac=0.0, temps=(1.0, 1.0))
    x = b.logits[0::2].astype(np.float64)
    p = np.exp(x - x.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    b.draft_probs = (2.0 * p).astype(np.float32)
    b.draft_ids = np.argmax(p, axis=1).astype(np.int32)
    ref = oracle.run(b)
    assert (ref["race_kind"] == oracle.RACE_FALLBACK).sum() > 10
    got = gpu_run(b)
    assert_parity(b, got, ref)


def test_inconsistent_batch_sets_error_and_context_recovers():
    import speculative_decoding_verification_rejection_gb300 as sv

    b = _custom(14, 4096, [2, 3, 1], "bf16", "noisy")
    ctx = sv.SpecVerify(8, 6, 4096, "bf16", True)
    bad = workloads.Batch(**{**b.__dict__})
    bad.cu_num_draft = np.array([0, 4, 3, 6], np.int32)       # decreasing
    got = gpu_run(bad, ctx, max_spec_len=6)
    assert got["error_word"] & sv.SV_ERR_BATCH
    assert np.all(got["num_sampled"] == 0) and np.all(got["sampled"] == -1)
    ok = gpu_run(b, ctx, max_spec_len=6)
    assert ok["error_word"] == 0
    assert_parity(b, ok, oracle.run(b, max_spec_len=6))
    ctx.close()


def test_host_side_errors_launch_nothing():
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    ctx = sv.SpecVerify(4, 3, 1024, "f32", False)
    b = workloads.workload(0)
    d = to_device(b)
    with pytest.raises(sv.SpecVerifyError) as e:     # draft probs given to a no-probs context
        ctx.run(d["logits"], d["draft_ids"], d["draft_probs"], d["cu_num_draft"], d["temperature"],
                d["is_greedy"], 0)
    assert e.value.status == sv.SV_EINVAL
    with pytest.raises(sv.SpecVerifyError) as e:     # more requests than the capacity
        sv.spec_verify_run(ctx.ctx, d["logits"], d["draft_ids"], None, d["cu_num_draft"],
                           d["temperature"], d["is_greedy"], 0, 0, 5, 12, 3,
                           torch.empty(5, 4, dtype=torch.int32, device="cuda"),
                           torch.empty(5, dtype=torch.int32, device="cuda"),
                           torch.empty(5, dtype=torch.int32, device="cuda"))
    assert e.value.status == sv.SV_ECAPACITY
    with pytest.raises(sv.SpecVerifyError) as e:     # NULL output
        sv.spec_verify_run(ctx.ctx, d["logits"], d["draft_ids"], None, d["cu_num_draft"],
                           d["temperature"], d["is_greedy"], 0, 0, 4, 12, 3, None, None, None)
    assert e.value.status == sv.SV_EINVAL
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.SpecVerify(4, 3, 1024, "f32", False, device=torch.cuda.device_count())
    assert e.value.status == sv.SV_EDEVICE
    # empty batch is a no-op
    sv.spec_verify_run(ctx.ctx, d["logits"], d["draft_ids"], None, d["cu_num_draft"],
                       d["temperature"], d["is_greedy"], 0, 0, 0, 0, 0, None, None, None)
    ctx.close()


def test_host_buffer_entry_point_matches():
    import speculative_decoding_verification_rejection_gb300 as sv

    b = workloads.workload(1)
    ctx = sv.SpecVerify(b.num_reqs, b.max_spec_len, b.vocab_size, "bf16", True)
    ctx.reserve_host_io()
    dev = gpu_run(b, ctx)
    n, k = b.num_reqs, b.max_spec_len
    sampled = np.empty((n, k + 1), np.int32)
    ns = np.empty(n, np.int32)
    nr = np.empty(n, np.int32)
    ctx.run_host(b.logits, b.draft_ids, b.draft_probs, b.cu_num_draft, b.temperature, b.is_greedy,
                 b.seed, sampled, ns, nr)
    np.testing.assert_array_equal(sampled, dev["sampled"])
    np.testing.assert_array_equal(ns, dev["num_sampled"])
    np.testing.assert_array_equal(nr, dev["num_rejected"])
    ctx.close()


def test_repeatable_and_profiled():
    import speculative_decoding_verification_rejection_gb300 as sv

    b = workloads.workload(2)
    ctx = sv.SpecVerify(b.num_reqs, b.max_spec_len, b.vocab_size, "bf16", False)
    ctx.set_profiling(True)
    a = gpu_run(b, ctx)
    c = gpu_run(b, ctx)
    for k in ("sampled", "num_sampled", "row_sumexp"):
        np.testing.assert_array_equal(a[k], c[k])
    ms, calls = ctx.get_profile()
    assert calls == 2 and ms["stats"] > 0 and ms["verify"] > 0 and ms["select"] >= 0
    ctx.close()


def test_cuda_graph_capture_and_replay():
    """spec_verify_run inside a captured CUDA graph: replays give the results of direct calls,
    also after new inputs are copied into the captured buffers."""
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    b1 = workloads.workload(1)
    b2 = _custom(15, b1.vocab_size, list(b1.cu_num_draft[1:] - b1.cu_num_draft[:-1]), "bf16", "noisy")
    ctx = sv.SpecVerify(b1.num_reqs, b1.max_spec_len, b1.vocab_size, "bf16", True)
    d = to_device(b1)
    n, k = b1.num_reqs, b1.max_spec_len
    outs = (torch.empty((n, k + 1), dtype=torch.int32, device="cuda"),
            torch.empty(n, dtype=torch.int32, device="cuda"),
            torch.empty(n, dtype=torch.int32, device="cuda"))

    def call():
        ctx.run(d["logits"], d["draft_ids"], d["draft_probs"], d["cu_num_draft"], d["temperature"],
                d["is_greedy"], b1.seed, out=outs)

    call()
    torch.cuda.synchronize()
    direct1 = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for o in outs:
        o.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    for a, c in zip(outs, direct1):
        assert torch.equal(a, c)
    # new inputs in the same buffers (same shapes and batch layout), replay again
    d2 = to_device(b2)
    for key in ("logits", "draft_ids", "draft_probs", "temperature", "is_greedy"):
        d[key].copy_(d2[key])
    g.replay()
    torch.cuda.synchronize()
    replayed2 = [o.clone() for o in outs]
    call()
    torch.cuda.synchronize()
    for a, c in zip(replayed2, outs):
        assert torch.equal(a, c)
    assert not torch.equal(replayed2[0], direct1[0])  # the new inputs were used
    del g
    ctx.close()


def test_host_entry_point_reads_page_locked_q_in_place():
    """run_host with page-locked inputs (q read in place by the kernels) matches the device path."""
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    b = workloads.workload(1)
    ctx = sv.SpecVerify(b.num_reqs, b.max_spec_len, b.vocab_size, "bf16", True)
    ctx.reserve_host_io()
    dev = gpu_run(b, ctx)
    n, k = b.num_reqs, b.max_spec_len
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    outs = [torch.empty((n, k + 1), dtype=torch.int32).pin_memory(),
            torch.empty(n, dtype=torch.int32).pin_memory(),
            torch.empty(n, dtype=torch.int32).pin_memory()]
    ctx.run_host(pin(b.logits.view(np.int16)), pin(b.draft_ids), pin(b.draft_probs),
                 pin(b.cu_num_draft), pin(b.temperature), pin(b.is_greedy), b.seed, *outs)
    np.testing.assert_array_equal(outs[0].numpy(), dev["sampled"])
    np.testing.assert_array_equal(outs[1].numpy(), dev["num_sampled"])
    np.testing.assert_array_equal(outs[2].numpy(), dev["num_rejected"])
    ctx.close()
