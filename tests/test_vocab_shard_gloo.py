"""Vocabulary-sharded verification over CPU ranks (gloo, world size 2 and 3): each rank holds a
column range of the logits and draft probabilities, and the two exchanges of
shard.sharded_verify (row statistics, then the best race key per request) must reproduce the
unsharded step. The per-rank arithmetic is the oracle's protocol side here (no GPU); what is
tested is the protocol and the host logic that drives the exchanges over torch.distributed."""
import os
import socket

import numpy as np
import pytest

import oracle
import workloads
from speculative_decoding_verification_rejection_gb300.shard import (VOCAB_ALIGN, sharded_verify,
                                                                     vocab_bounds)


def _batch(kind):
    rng = np.random.default_rng(5)
    n = 29
    K = rng.integers(0, 6, n)
    q_mode = {"probs": "noisy", "ids": "none"}[kind]
    return workloads.make_batch(name="vshard", data_seed=41, verify_seed=99, K=K, vocab_size=1000,
                                logits_dtype="bf16", sigma=2.0, zipf_coef=0.8, q_mode=q_mode,
                                q_noise=1.5, p_argmax=0.6,
                                temperature=rng.uniform(0.4, 1.4, n).astype(np.float32),
                                greedy=(rng.random(n) < 0.25).astype(np.uint8))


def _rank_main(rank, world, port, kind, out_path):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _batch(kind)
        lo, hi = vocab_bounds(b.vocab_size, world)[rank]
        backend = oracle.ShardOracle(b, lo, hi - lo)

        def all_gather(rec):
            t = torch.from_numpy(np.ascontiguousarray(rec).view(np.uint8).copy())
            parts = [torch.empty_like(t) for _ in range(world)]
            dist.all_gather(parts, t)
            return np.stack([p.numpy().view(rec.dtype) for p in parts])

        sampled, ns, nr = sharded_verify(backend, all_gather, world, b.max_spec_len)
        if rank == 0:
            np.savez(out_path, sampled=sampled, num_sampled=ns, num_rejected=nr)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world,kind", [(2, "probs"), (3, "ids")])
def test_gloo_ranks_reproduce_the_unsharded_step(tmp_path, world, kind):
    import torch.multiprocessing as mp

    oracle.build()
    out = str(tmp_path / "out.npz")
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, kind, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    got = np.load(out)
    full = oracle.run(_batch(kind))
    np.testing.assert_array_equal(got["sampled"], full["sampled"])
    np.testing.assert_array_equal(got["num_sampled"], full["num_sampled"])
    np.testing.assert_array_equal(got["num_rejected"], full["num_rejected"])


def test_vocab_bounds():
    for V in (1, 63, 64, 1000, 151936, 129280):
        for world in (1, 2, 3, 4, 8):
            b = vocab_bounds(V, world)
            assert len(b) == world and b[0][0] == 0 and b[-1][1] == V
            assert all(lo % VOCAB_ALIGN == 0 or lo == V for lo, _ in b)
            assert all(b[k][1] == b[k + 1][0] for k in range(world - 1))
            assert sum(hi - lo for lo, hi in b) == V


@pytest.mark.parametrize("c", [0, 1, 2, 4])
def test_in_process_shards_match_the_unsharded_oracle(c):
    """The protocol with the exchange done in-process, on the named workloads (shorter)."""
    b = workloads.workload(c, num_reqs=24)
    full = oracle.run(b)
    for world in (2, 4):
        sides = [oracle.ShardOracle(b, lo, hi - lo) for lo, hi in vocab_bounds(b.vocab_size, world)
                 if hi > lo]
        w = len(sides)
        st = np.stack([s.stats() for s in sides])
        rc = np.stack([s.race(st, w) for s in sides])
        sampled, ns, nr = sides[0].finish(rc, w, b.max_spec_len)
        np.testing.assert_array_equal(sampled, full["sampled"])
        np.testing.assert_array_equal(ns, full["num_sampled"])
        np.testing.assert_array_equal(nr, full["num_rejected"])
