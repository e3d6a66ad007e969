"""Run by tests/test_gpu_debug_bounds.py in a child process whose library is the bounds-checked
build (SPEC_VERIFY_DEBUG_BOUNDS=1): every global load and store of every kernel is checked
against the arrays of its call, an access outside them is skipped and sets SV_ERR_BOUNDS in the
error word. Small cases cover every entry point and input mode; each must match the oracle and
leave the bit clear. A positive control then leaves the last bytes of the logits out of the
registered ranges (the memory itself is valid) and the bit must appear. Prints OK at the end."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
import workloads  # noqa: E402
from _parity import assert_parity, gpu_run, to_device  # noqa: E402


def small(seed, V, Ks, dtype, q_mode, greedy_frac=0.25):
    rng = np.random.default_rng(seed)
    n = len(Ks)
    return workloads.make_batch(name=f"dbg{seed}", data_seed=seed, verify_seed=seed + 99, K=Ks,
                                vocab_size=V, logits_dtype=dtype, sigma=2.0, zipf_coef=0.7,
                                n_boost=3, boost=4.0, q_mode=q_mode, q_noise=1.2, p_argmax=0.6,
                                temperature=rng.uniform(0.4, 1.4, n).astype(np.float32),
                                greedy=(rng.random(n) < greedy_frac).astype(np.uint8))


def check(b, label):
    got = gpu_run(b)
    assert_parity(b, got, oracle.run(b))
    assert not got["error_word"] & sv.SV_ERR_BOUNDS, f"{label}: out-of-bounds access"
    print(f"{label}: clean", flush=True)


def run_noalloc(b):
    import torch

    d = to_device(b)
    n, nd, k = b.num_reqs, b.num_draft_tokens, b.max_spec_len
    outs = [torch.empty((n, k + 1), dtype=torch.int32, device="cuda"),
            torch.empty(n, dtype=torch.int32, device="cuda"),
            torch.empty(n, dtype=torch.int32, device="cuda")]
    sv.spec_verify_run_noalloc(d["logits"], b.logits_dtype, b.vocab_size, d["draft_ids"],
                               d["draft_probs"], d["cu_num_draft"], d["temperature"], d["is_greedy"],
                               b.seed, 0, n, nd, k, *outs)
    torch.cuda.synchronize()
    ref = oracle.run(b)
    np.testing.assert_array_equal(outs[0].cpu().numpy(), ref["sampled"])
    assert not sv.spec_verify_noalloc_last_error() & sv.SV_ERR_BOUNDS, "noalloc: out-of-bounds access"
    print("noalloc: clean", flush=True)


def run_host(b):
    ctx = sv.SpecVerify(b.num_reqs, b.max_spec_len, b.vocab_size, b.logits_dtype,
                        b.draft_probs is not None)
    ctx.reserve_host_io()
    n, k = b.num_reqs, b.max_spec_len
    out = (np.empty((n, k + 1), np.int32), np.empty(n, np.int32), np.empty(n, np.int32))
    ctx.run_host(np.ascontiguousarray(b.logits), b.draft_ids, b.draft_probs, b.cu_num_draft,
                 b.temperature, b.is_greedy, b.seed, *out)
    np.testing.assert_array_equal(out[0], oracle.run(b)["sampled"])
    assert not ctx.last_error() & sv.SV_ERR_BOUNDS, "host entry point: out-of-bounds access"
    ctx.close()
    print("host entry point: clean", flush=True)


def run_shards(b, world):
    import torch

    from speculative_decoding_verification_rejection_gb300.shard import ShardBackend, vocab_bounds

    dev = "cuda:0"
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dt)).to(dev)  # noqa: E731
    ids, cu = t(b.draft_ids, np.int32), t(b.cu_num_draft, np.int32)
    T, g = t(b.temperature, np.float32), t(b.is_greedy, np.uint8)
    logits = np.ascontiguousarray(b.logits)
    sides, ctxs = [], []
    for lo, hi in [x for x in vocab_bounds(b.vocab_size, world) if x[1] > x[0]]:
        sl = np.ascontiguousarray(logits[:, lo:hi])
        lt = torch.from_numpy(sl.view(np.int16) if sl.dtype == np.uint16 else sl).to(dev)
        q = None if b.draft_probs is None else t(np.asarray(b.draft_probs)[:, lo:hi], np.float32)
        ctx = sv.SpecVerify(b.num_reqs, b.max_spec_len, hi - lo, b.logits_dtype,
                            b.draft_probs is not None)
        ctxs.append(ctx)
        sides.append(ShardBackend(ctx, lo, b.vocab_size, lt, ids, q, cu, T, g, b.seed,
                                  max_spec_len=b.max_spec_len))
    w = len(sides)
    all_stats = torch.cat([s.stats() for s in sides])
    all_races = torch.cat([s.race(all_stats, w) for s in sides])
    sampled, _, _ = sides[0].finish(all_races, w, b.max_spec_len)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(sampled.cpu().numpy(), oracle.run(b)["sampled"])
    for c in ctxs:
        assert not c.last_error() & sv.SV_ERR_BOUNDS, "shards: out-of-bounds access"
        c.close()
    print(f"{world} vocabulary shards: clean", flush=True)


if __name__ == "__main__":
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    assert sv.DEBUG_BOUNDS and sv.LIB_PATH.endswith("libspecverify_debug.so")
    assert torch.cuda.is_available()
    sv.lib()
    check(workloads.workload(0), "workload 0")
    for seed, V, Ks, dtype, q_mode in ((301, 1000, [3, 0, 5, 1, 2], "f32", "noisy"),
                                       (302, 1001, [2, 2, 0, 6, 1], "bf16", "none"),
                                       (303, 9001, [3, 2, 4, 0], "bf16", "indep"),
                                       (304, 4004, [2, 4, 0, 3], "bf16", "logits"),
                                       (305, 7, [3, 1, 0, 2], "f32", "noisy")):
        check(small(seed, V, Ks, dtype, q_mode), f"{dtype} {q_mode} V={V}")
    b = small(306, 3001, [4, 4, 2, 0, 3, 4], "bf16", "noisy")
    workloads.add_penalty(b, 306, history=(20, 80), top_n=20, extra_rows=2, shuffle_rows=True)
    check(b, "frequency penalty")
    rng = np.random.default_rng(307)
    b.top_k = rng.choice(np.array([0, 20, 300], np.int32), b.num_reqs).astype(np.int32)
    b.top_p = rng.choice(np.array([0.8, 1.0], np.float32), b.num_reqs).astype(np.float32)
    check(b, "penalty + top-k / top-p")
    b.fp64_gumbel = True
    check(b, "penalty + top-k / top-p + fp64 races")
    b = small(308, 2003, [3, 2, 4, 1], "f32", "noisy")
    b.synthetic_rates = np.array([0.9, 0.5, 0.3], np.float32)
    b.partial_prefill = np.array([0, 1, 0, 0], np.uint8)
    check(b, "synthetic acceptance + chunked prefill")
    run_noalloc(small(309, 5003, [2, 3, 0, 4], "bf16", "noisy"))
    run_host(small(310, 3000, [2, 3, 1], "f32", "noisy"))
    run_shards(small(311, 4096 + 64 * 3, [2, 0, 3, 1], "bf16", "noisy"), 3)
    # positive control: the registered logits range lacks its last 64 bytes (the memory is
    # still there); the statistics kernel reads them, so the check must fire, and the context
    # must stay usable afterwards
    os.environ["SV_DEBUG_SHRINK"] = "64"
    b = workloads.workload(0)
    got = gpu_run(b)
    del os.environ["SV_DEBUG_SHRINK"]
    assert got["error_word"] & sv.SV_ERR_BOUNDS, "the check did not fire"
    print("positive control: fired", flush=True)
    check(workloads.workload(0), "after the control")
    print("OK", flush=True)
