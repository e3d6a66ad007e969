"""Request sharding over CPU ranks (gloo, world size 2): each rank verifies its contiguous request
range with req_index_base = its first request; the gathered outputs must equal the whole batch's.
The verification itself is the oracle here (no GPU); what is tested is the host logic that splits
a batch, keys the shards and joins their outputs."""
import os
import socket

import numpy as np
import pytest

import oracle
import workloads
from speculative_decoding_verification_rejection_gb300.shard import make_shard, shard_bounds, shards


def _sub_batch(b, sh):
    return workloads.Batch(
        name="shard", logits=b.logits[sh.row_lo:sh.row_hi], logits_dtype=b.logits_dtype,
        vocab_size=b.vocab_size, draft_ids=b.draft_ids[sh.draft_lo:sh.draft_hi],
        draft_probs=None if b.draft_probs is None else b.draft_probs[sh.draft_lo:sh.draft_hi],
        cu_num_draft=sh.cu_num_draft, temperature=b.temperature[sh.lo:sh.hi],
        is_greedy=b.is_greedy[sh.lo:sh.hi], seed=b.seed)


def _batch():
    rng = np.random.default_rng(3)
    K = rng.integers(0, 6, 37)
    return workloads.make_batch(name="ragged", data_seed=31, verify_seed=77, K=K, vocab_size=301,
                                logits_dtype="bf16", sigma=2.0, q_mode="noisy", q_noise=1.5,
                                temperature=rng.uniform(0.4, 1.4, 37).astype(np.float32),
                                greedy=(rng.random(37) < 0.25).astype(np.uint8))


def _rank_main(rank, world, port, out_path):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _batch()
        sh = shards(b.cu_num_draft, world)[rank]
        kmax = b.max_spec_len
        got = oracle.run(_sub_batch(b, sh), max_spec_len=kmax, req_index_base=sh.lo)
        parts = [None] * world
        dist.all_gather_object(parts, (sh.lo, got["sampled"], got["num_sampled"],
                                       got["num_rejected"], sh.num_rows))
        if rank == 0:
            parts.sort(key=lambda p: p[0])
            np.savez(out_path, sampled=np.concatenate([p[1] for p in parts]),
                     num_sampled=np.concatenate([p[2] for p in parts]),
                     num_rejected=np.concatenate([p[3] for p in parts]),
                     rows=np.array([p[4] for p in parts]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_reproduce_the_whole_batch(tmp_path):
    import torch.multiprocessing as mp

    oracle.build()
    out = str(tmp_path / "joined.npz")
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    joined = np.load(out)
    b = _batch()
    full = oracle.run(b)
    np.testing.assert_array_equal(joined["sampled"], full["sampled"])
    np.testing.assert_array_equal(joined["num_sampled"], full["num_sampled"])
    np.testing.assert_array_equal(joined["num_rejected"], full["num_rejected"])
    assert abs(int(joined["rows"][0]) - int(joined["rows"][1])) <= b.max_spec_len + 1


def test_shard_bounds_cover_balance_and_handle_small_batches():
    rng = np.random.default_rng(0)
    for world in (1, 2, 3, 8):
        K = rng.integers(0, 6, 50)
        cu = np.concatenate([[0], np.cumsum(K)]).astype(np.int32)
        b = shard_bounds(cu, world)
        assert len(b) == world and b[0][0] == 0 and b[-1][1] == 50
        assert all(lo <= hi for lo, hi in b) and all(b[k][1] == b[k + 1][0] for k in range(world - 1))
        rows = [make_shard(cu, lo, hi).num_rows for lo, hi in b]
        assert sum(rows) == int(cu[-1]) + 50
        assert max(rows) - min(rows) <= 2 * (K.max() + 1)
    b = shard_bounds(np.array([0, 2, 3], np.int32), 4)  # fewer requests than ranks
    assert len(b) == 4 and sum(hi - lo for lo, hi in b) == 2
    sh = make_shard(np.array([0, 2, 3, 7], np.int32), 1, 3)
    assert (sh.row_lo, sh.row_hi, sh.draft_lo, sh.draft_hi) == (3, 10, 2, 7)
    np.testing.assert_array_equal(sh.cu_num_draft, [0, 1, 5])
