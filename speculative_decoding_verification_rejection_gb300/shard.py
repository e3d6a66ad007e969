"""Request sharding across ranks (host logic, no device code).

Requests are independent: each one is verified from its own logit rows and draws its own random
numbers ([MTP-eagle] _rejection_sample_kernel runs one program per request). A batch therefore
splits into contiguous request ranges with no exchange between them. Rank k verifies requests
[lo, hi) from their own rows with ``req_index_base = lo``, which keys every draw exactly as in
the whole batch, and the ranks' outputs concatenate to the whole batch's outputs.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Shard:
    """Requests [lo, hi) of a batch and where their data sits in the whole batch's arrays."""
    lo: int
    hi: int
    row_lo: int    # first logit row (cu_num_draft[lo] + lo)
    row_hi: int    # one past the last logit row
    draft_lo: int  # first draft token (cu_num_draft[lo])
    draft_hi: int
    cu_num_draft: np.ndarray  # the shard's own prefix sums, starting at 0

    @property
    def num_reqs(self) -> int:
        return self.hi - self.lo

    @property
    def num_rows(self) -> int:
        return self.row_hi - self.row_lo


def shard_bounds(cu_num_draft, world_size: int) -> list[tuple[int, int]]:
    """Contiguous request ranges [lo, hi), one per rank, balanced by logit rows (every row is V
    logits, the dominant bytes): rank k's range ends at the first request boundary at or after
    k + 1 world_size-ths of the rows. Ranges may be empty when there are fewer requests than ranks."""
    cu = np.asarray(cu_num_draft, dtype=np.int64)
    n = cu.shape[0] - 1
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    rows_before = cu + np.arange(n + 1)  # rows of requests 0 .. i-1
    total = int(rows_before[-1])
    cuts = [0]
    for k in range(1, world_size):
        target = (total * k + world_size - 1) // world_size
        cut = int(np.searchsorted(rows_before, target, side="left"))
        cuts.append(min(max(cut, cuts[-1]), n))
    cuts.append(n)
    return list(zip(cuts[:-1], cuts[1:]))


def make_shard(cu_num_draft, lo: int, hi: int) -> Shard:
    cu = np.asarray(cu_num_draft, dtype=np.int64)
    return Shard(lo=lo, hi=hi, row_lo=int(cu[lo] + lo), row_hi=int(cu[hi] + hi),
                 draft_lo=int(cu[lo]), draft_hi=int(cu[hi]),
                 cu_num_draft=(cu[lo:hi + 1] - cu[lo]).astype(np.int32))


def shards(cu_num_draft, world_size: int) -> list[Shard]:
    return [make_shard(cu_num_draft, lo, hi) for lo, hi in shard_bounds(cu_num_draft, world_size)]


# ---------------------------------------------------------------------------------------------
# Vocabulary sharding: every rank holds a column range of every logit row (a tensor-parallel LM
# head's output), and two small exchanges replace gathering the rows.
# ---------------------------------------------------------------------------------------------
VOCAB_ALIGN = 64  # shard boundaries on race-clock groups of 64 tokens


def vocab_bounds(vocab_size: int, world_size: int) -> list[tuple[int, int]]:
    """Column ranges [v0, v1), one per rank, each starting on a multiple of 64 tokens (a race
    clock group never straddles two ranks), as even as that allows; trailing ranks may be empty."""
    if world_size < 1 or vocab_size < 1:
        raise ValueError("world_size and vocab_size must be >= 1")
    step = -(-vocab_size // world_size)
    step = -(-step // VOCAB_ALIGN) * VOCAB_ALIGN
    return [(min(vocab_size, r * step), min(vocab_size, (r + 1) * step)) for r in range(world_size)]


def sharded_verify(backend, all_gather, world_size: int, max_spec_len: int):
    """One verification step over vocabulary shards, on one rank.

    backend: this rank's side of the protocol, with
      stats()                      -> this rank's statistics record of every logit row
      race(all_stats, world_size)  -> this rank's race record of every request, given the
                                      statistics of all ranks (rank-major)
      finish(all_races, world_size, max_spec_len) -> (sampled, num_sampled, num_rejected)
    all_gather(x): the records of every rank stacked in rank order (the exchange).

    Exchange 1 carries, per row, the shard's largest logit with its first index, its sum of
    exponentials and, from the shard holding the row's draft token, that token's logit and draft
    probability: every rank then combines the same numbers in the same order and takes the same
    acceptance decisions. Exchange 2 carries, per request, each shard's best race key at the row
    of the first rejection (residual or exclusion race, and the race over p for the fallback and
    the bonus); the largest key over the shards is the winner of the whole row, since every key
    is computed with the combined maximum and sum and the global race clocks.
    """
    all_stats = all_gather(backend.stats())
    all_races = all_gather(backend.race(all_stats, world_size))
    return backend.finish(all_races, world_size, max_spec_len)


class ShardBackend:
    """This rank's side of sharded_verify on its GPU: device tensors for its columns
    [v0, v0 + Vs) of the logits (and draft probabilities); records are uint8 device tensors
    (24 bytes per row, then per request) ready for an all-gather."""

    def __init__(self, ctx, v0: int, vocab_size: int, logits_shard, draft_ids, draft_probs_shard,
                 cu_num_draft, temperature, is_greedy, seed: int, req_index_base: int = 0,
                 max_spec_len: int | None = None, stream=None):
        from . import SHARD_RECORD_BYTES
        self.ctx, self.v0, self.V = ctx, int(v0), int(vocab_size)
        self.logits, self.ids, self.q = logits_shard, draft_ids, draft_probs_shard
        self.cu, self.T, self.g = cu_num_draft, temperature, is_greedy
        self.seed, self.base, self.stream = seed, req_index_base, stream
        self.n = cu_num_draft.numel() - 1
        self.nd = draft_ids.numel()
        self.kmax = ctx.max_spec_len if max_spec_len is None else max_spec_len
        self.rec = SHARD_RECORD_BYTES

    def stats(self):
        import torch
        from . import spec_verify_shard_stats
        out = torch.empty((self.nd + self.n) * self.rec, dtype=torch.uint8, device=self.logits.device)
        spec_verify_shard_stats(self.ctx.ctx, self.logits, self.v0, self.ids, self.q, self.cu, self.T,
                                self.g, self.n, self.nd, self.kmax, out, cuda_stream=self.stream)
        return out

    def race(self, all_stats, world_size: int):
        import torch
        from . import spec_verify_shard_race
        out = torch.empty(self.n * self.rec, dtype=torch.uint8, device=self.logits.device)
        spec_verify_shard_race(self.ctx.ctx, self.logits, self.v0, self.V, all_stats.contiguous(),
                               world_size, self.ids, self.q, self.cu, self.T, self.g, self.seed,
                               self.base, self.n, self.nd, self.kmax, out, cuda_stream=self.stream)
        return out

    def finish(self, all_races, world_size: int, max_spec_len: int):
        import torch
        from . import spec_verify_shard_finish
        dev = self.logits.device
        sampled = torch.empty((self.n, max_spec_len + 1), dtype=torch.int32, device=dev)
        ns = torch.empty(self.n, dtype=torch.int32, device=dev)
        nr = torch.empty(self.n, dtype=torch.int32, device=dev)
        spec_verify_shard_finish(self.ctx.ctx, all_races.contiguous(), world_size, self.ids, self.cu,
                                 self.n, max_spec_len, sampled, ns, nr, cuda_stream=self.stream)
        return sampled, ns, nr


def nccl_all_gather(group=None):
    """The exchange of sharded_verify over torch.distributed: the ranks' byte records stacked
    in rank order."""
    def gather(rec):
        import torch
        import torch.distributed as dist
        world = dist.get_world_size(group)
        out = torch.empty(world * rec.numel(), dtype=rec.dtype, device=rec.device)
        dist.all_gather_into_tensor(out, rec.contiguous(), group=group)
        return out
    return gather
