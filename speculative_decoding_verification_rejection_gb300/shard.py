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
