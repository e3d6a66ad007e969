"""Seeded synthetic inputs for the speculative-decoding verification sampler.

Shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``. The arrays are built by
``gen.c`` (compiled on first use with gcc; OpenMP when available) from a counter-based
hash, so every value is a pure function of the data seed and its position.

The five named workloads follow the shapes and value distributions of the verification
step described on the pages (target logits at K draft positions plus one bonus position
per request, an optional draft distribution q, and the draft token ids):

====  ============================================================================
 0    tiny: 4 requests, K=3, V=1024, fp32 logits N(0, 2^2), q = softmax(target + N(0,1)),
      draft ids drawn from q, T = 1, all random
 1    64 requests, K=4, V=32000, bf16 logits N(0, 3^2) with 5 tokens boosted by +8,
      q = softmax(target + N(0, 1.5^2)), T ~ U[0.5, 1.2], 16 greedy requests
 2    128 requests, K_i ~ U{0..5}, V=128256, bf16 Zipf logits -1.1 ln(rank) + N(0, 0.5^2),
      no q (draft ids only): 70% equal the target argmax, else uniform; T = 0.8
 3    256 requests, K=5, V=151936, bf16 logits N(0, 2.5^2) - 1.1 ln(rank),
      q = softmax(target + N(0, 2^2)), T = 1  (the bandwidth workload)
 4    512 requests: 256 random K=3, 128 greedy K=3, 128 non-speculative K=0; V=129280,
      fp32 logits N(0, 2^2) with 10 tokens boosted by +6, q from an independent N(0, 2^2)
      draw, T ~ U[0.3, 1.5] for the random and non-speculative requests
====  ============================================================================

The data seed and the verification seed of workload c are both c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libsvgen.so")
_lib = None

# Stream tags of the generator hash (one per drawn quantity).
_S_LOGITS, _S_Q, _S_IDS, _S_TEMP, _S_K, _S_GROUP = 1000, 2000, 3000, 4000, 5000, 6000


def build(force: bool = False) -> str:
    """Compile gen.c into libsvgen.so next to it (atomic replace). Returns the path."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=gnu11", _SRC, "-o", tmp, "-lm"]
    try:
        r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
        if r.returncode != 0:  # no OpenMP runtime: the generator is still correct, just serial
            subprocess.run(base, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB_PATH)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, d, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_int
        vp = ctypes.c_void_p
        lib.gen_uniform.argtypes = [u64, u64, i64, vp]
        lib.gen_target_logits.argtypes = [u64, u64, i64, i64, d, d, i32, d, i32, vp]
        lib.gen_draft_probs.argtypes = [u64, u64, i64, i64, vp, vp, i32, d, i32, d, vp]
        lib.gen_sample_from_q.argtypes = [u64, u64, i64, i64, vp, vp]
        lib.gen_draft_logits.argtypes = [u64, u64, i64, i64, vp, vp, i32, d, vp]
        lib.gen_sample_from_logits.argtypes = [u64, u64, i64, i64, vp, i32, vp, vp]
        lib.gen_argmax_or_uniform.argtypes = [u64, u64, i64, i64, vp, vp, i32, d, vp]
        for f in ("gen_uniform", "gen_target_logits", "gen_draft_probs", "gen_sample_from_q",
                  "gen_argmax_or_uniform"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        _load().gen_uniform(seed, stream, n, _ptr(out))
    return out


def shuffled(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n) (Fisher-Yates on the generator's uniforms)."""
    u = uniform(seed, stream, n)
    p = np.arange(n)
    for k in range(n - 1, 0, -1):
        j = min(int(u[k] * (k + 1)), k)
        p[k], p[j] = p[j], p[k]
    return p


@dataclass
class Batch:
    """One verification batch, host-resident (numpy)."""

    name: str
    logits: np.ndarray          # [R, V] uint16 (bf16 bits) or float32
    logits_dtype: str           # "bf16" | "f32"
    vocab_size: int
    draft_ids: np.ndarray       # [N_d] int32
    draft_probs: np.ndarray | None  # [N_d, V] float32 or None (draft ids only)
    cu_num_draft: np.ndarray    # [num_reqs + 1] int32
    temperature: np.ndarray     # [num_reqs] float32
    is_greedy: np.ndarray       # [num_reqs] uint8
    seed: int
    meta: dict = field(default_factory=dict)
    # [N_d, V] draft logits in the logits' type (draft-logits mode: q = softmax(dl / T)), or None
    draft_logits: np.ndarray | None = None
    # [num_reqs] uint8: requests still in a chunked prefill (they report no token), or None
    partial_prefill: np.ndarray | None = None
    # synthetic acceptance: unconditional rate per draft position (verifier setting), or None
    synthetic_rates: np.ndarray | None = None
    # logits processors: [num_reqs] float32 frequency penalty with [rows, V] int32 output token
    # counts (row counts_row[i], or i, per request); [num_reqs] int32 top_k, float32 top_p
    frequency_penalty: np.ndarray | None = None
    output_bin_counts: np.ndarray | None = None
    counts_row: np.ndarray | None = None
    top_k: np.ndarray | None = None
    top_p: np.ndarray | None = None
    # race noise drawn in binary64 (the fp64 Gumbel option, a per-call verifier setting)
    fp64_gumbel: bool = False

    @property
    def num_reqs(self) -> int:
        return int(self.cu_num_draft.shape[0] - 1)

    @property
    def num_draft_tokens(self) -> int:
        return int(self.cu_num_draft[-1])

    @property
    def num_rows(self) -> int:
        return self.num_draft_tokens + self.num_reqs

    @property
    def max_spec_len(self) -> int:
        k = np.diff(self.cu_num_draft)
        return int(k.max()) if k.size else 0

    @property
    def elem_bytes(self) -> int:
        return 2 if self.logits_dtype == "bf16" else 4

    def random_draft_rows(self) -> int:
        """Draft rows of requests that sample (non-greedy): the rows whose q a full pass reads."""
        k = np.diff(self.cu_num_draft).astype(np.int64)
        greedy = (self.is_greedy != 0) | ~(self.temperature > 0)
        return int(k[~greedy].sum())

    def bytes_full(self) -> int:
        """Every logit row once plus every sampling request's q rows once."""
        b = self.num_rows * self.vocab_size * self.elem_bytes
        if self.draft_probs is not None:
            b += self.random_draft_rows() * self.vocab_size * 4
        if self.draft_logits is not None:
            b += self.random_draft_rows() * self.vocab_size * self.elem_bytes
        return b


def _row_of_qrow(cu: np.ndarray) -> np.ndarray:
    k = np.diff(cu)
    req = np.repeat(np.arange(k.size, dtype=np.int64), k)
    return (np.arange(int(cu[-1]), dtype=np.int64) + req).astype(np.int32)


def make_batch(*, name: str, data_seed: int, verify_seed: int, K, vocab_size: int,
               logits_dtype: str = "f32", sigma: float = 2.0, zipf_coef: float = 0.0,
               n_boost: int = 0, boost: float = 0.0, q_mode: str = "noisy", q_noise: float = 1.0,
               q_indep_sigma: float = 2.0, p_argmax: float = 0.7, temperature=1.0,
               greedy=None) -> Batch:
    """Build a batch from a recipe.

    K: sequence of per-request draft lengths.
    q_mode: "noisy" (q = softmax(target + q_noise * N)), "indep" (q = softmax(q_indep_sigma * N)),
            "logits" (draft logits = target + q_noise * N in the logits' type, ids drawn from
            softmax(draft logits / T) of the request), or "none" (draft ids only: argmax with
            probability p_argmax, else uniform).
    temperature: float or per-request array. greedy: None or per-request bool array.
    """
    lib = _load()
    if np.isscalar(K):
        raise ValueError("pass K as a per-request sequence")
    Ks = np.asarray(K, dtype=np.int64)
    num_reqs = Ks.size
    cu = np.zeros(num_reqs + 1, dtype=np.int32)
    cu[1:] = np.cumsum(Ks)
    n_d = int(cu[-1])
    R = n_d + num_reqs
    V = int(vocab_size)
    bf16 = logits_dtype == "bf16"
    logits = np.empty((R, V), dtype=np.uint16 if bf16 else np.float32)
    if R:
        lib.gen_target_logits(data_seed, _S_LOGITS, R, V, sigma, zipf_coef, n_boost, boost,
                              int(bf16), _ptr(logits))
    src = _row_of_qrow(cu)
    ids = np.zeros(n_d, dtype=np.int32)
    q = None
    if q_mode in ("noisy", "indep"):
        q = np.empty((n_d, V), dtype=np.float32)
        if n_d:
            lib.gen_draft_probs(data_seed, _S_Q, n_d, V, _ptr(src), _ptr(logits), int(bf16),
                                q_noise, int(q_mode == "indep"), q_indep_sigma, _ptr(q))
            lib.gen_sample_from_q(data_seed, _S_IDS, n_d, V, _ptr(q), _ptr(ids))
    elif q_mode == "logits":
        temp_req = np.broadcast_to(np.asarray(temperature, dtype=np.float32), (num_reqs,))
        g_req = np.zeros(num_reqs, np.uint8) if greedy is None else np.asarray(greedy, np.uint8)
        dl = np.empty((n_d, V), dtype=np.uint16 if bf16 else np.float32)
        if n_d:
            lib.gen_draft_logits(data_seed, _S_Q, n_d, V, _ptr(src), _ptr(logits), int(bf16),
                                 q_noise, _ptr(dl))
            req_of_qrow = np.repeat(np.arange(num_reqs), Ks)
            t = temp_req[req_of_qrow].astype(np.float64)
            inv = np.where((g_req[req_of_qrow] != 0) | ~(t > 0), 1.0, 1.0 / np.where(t > 0, t, 1.0))
            inv = np.ascontiguousarray(inv, dtype=np.float64)
            lib.gen_sample_from_logits(data_seed, _S_IDS, n_d, V, _ptr(dl), int(bf16), _ptr(inv),
                                       _ptr(ids))
    elif q_mode == "none":
        if n_d:
            lib.gen_argmax_or_uniform(data_seed, _S_IDS, n_d, V, _ptr(src), _ptr(logits),
                                      int(bf16), p_argmax, _ptr(ids))
    else:
        raise ValueError(q_mode)
    temp = np.broadcast_to(np.asarray(temperature, dtype=np.float32), (num_reqs,)).copy()
    g = np.zeros(num_reqs, dtype=np.uint8) if greedy is None else np.asarray(greedy, dtype=np.uint8)
    return Batch(name=name, logits=logits, logits_dtype=logits_dtype, vocab_size=V, draft_ids=ids,
                 draft_probs=q, cu_num_draft=cu, temperature=temp, is_greedy=g, seed=verify_seed,
                 draft_logits=dl if q_mode == "logits" else None)


def add_penalty(b: Batch, seed: int, *, history=(50, 500), top_share=0.5, top_n=50,
                penalty=(-0.5, 1.5), extra_rows: int = 0, shuffle_rows: bool = False) -> Batch:
    """Give a batch a frequency penalty: per request a token history of U{history} tokens, each
    with probability top_share one of the top_n logits of the request's first row (the tokens a
    model tends to repeat), else uniform over the vocabulary; output_bin_counts = the history's
    counts; penalty ~ U(penalty). extra_rows unused count rows are added, and with shuffle_rows
    the requests' rows are permuted (counts_row maps them)."""
    rng = np.random.default_rng([seed, 0x5EED])
    n, V = b.num_reqs, b.vocab_size
    rows = n + extra_rows
    counts = np.zeros((rows, V), np.int32)
    perm = rng.permutation(rows)[:n] if shuffle_rows else np.arange(n)
    logits = b.logits
    for i in range(n):
        r0 = int(b.cu_num_draft[i]) + i
        row = logits[r0]
        vals = (row.astype(np.uint32) << 16).view(np.float32) if row.dtype == np.uint16 else row
        top = np.argsort(-vals, kind="stable")[:top_n]
        h = int(rng.integers(history[0], history[1] + 1))
        pick_top = rng.random(h) < top_share
        toks = np.where(pick_top, top[rng.integers(0, top.size, h)], rng.integers(0, V, h))
        np.add.at(counts[perm[i]], toks, 1)
    b.output_bin_counts = counts
    b.counts_row = perm.astype(np.int32) if shuffle_rows else None
    b.frequency_penalty = rng.uniform(*penalty, n).astype(np.float32)
    return b


WORKLOADS = {
    0: "tiny: 4 req, K=3, V=1024, fp32, q noisy, T=1",
    1: "64 req, K=4, V=32000, bf16 boosted, q noisy, T~U[0.5,1.2], 25% greedy",
    2: "128 req, K~U{0..5}, V=128256, bf16 Zipf, draft ids only, T=0.8",
    3: "256 req, K=5, V=151936, bf16 N(0,2.5^2)+Zipf, fp32 q, T=1",
    4: "512 req mixed (256 random K=3, 128 greedy K=3, 128 K=0), V=129280, fp32, indep q",
}


def workload(c: int, num_reqs: int | None = None, *, draft_logits: bool = False) -> Batch:
    """Named workload c (0..4). num_reqs, if given, keeps only the first num_reqs requests
    of the recipe (same per-request draws), for bounded samples. draft_logits=True gives the
    draft model's logits (target + q_noise * N, in the logits' type) instead of probabilities,
    for the recipes that have a draft distribution."""
    seed = c
    if c == 0:
        n = 4
        b = dict(K=[3] * n, vocab_size=1024, logits_dtype="f32", sigma=2.0, q_mode="noisy",
                 q_noise=1.0, temperature=1.0)
    elif c == 1:
        n = 64
        greedy = np.zeros(n, dtype=np.uint8)
        greedy[shuffled(seed, _S_GROUP, n)[: n // 4]] = 1
        temp = (0.5 + 0.7 * uniform(seed, _S_TEMP, n)).astype(np.float32)
        b = dict(K=[4] * n, vocab_size=32000, logits_dtype="bf16", sigma=3.0, n_boost=5, boost=8.0,
                 q_mode="noisy", q_noise=1.5, temperature=temp, greedy=greedy)
    elif c == 2:
        n = 128
        Ks = np.minimum((uniform(seed, _S_K, n) * 6).astype(np.int64), 5)
        b = dict(K=Ks, vocab_size=128256, logits_dtype="bf16", sigma=0.5, zipf_coef=1.1,
                 q_mode="none", p_argmax=0.7, temperature=0.8)
    elif c == 3:
        n = 256
        b = dict(K=[5] * n, vocab_size=151936, logits_dtype="bf16", sigma=2.5, zipf_coef=1.1,
                 q_mode="noisy", q_noise=2.0, temperature=1.0)
    elif c == 4:
        n = 512
        perm = shuffled(seed, _S_GROUP, n)
        kind = np.zeros(n, dtype=np.int64)          # 0 random, 1 greedy, 2 non-speculative
        kind[perm[256:384]] = 1
        kind[perm[384:]] = 2
        Ks = np.where(kind == 2, 0, 3)
        temp = (0.3 + 1.2 * uniform(seed, _S_TEMP, n)).astype(np.float32)
        b = dict(K=Ks, vocab_size=129280, logits_dtype="f32", sigma=2.0, n_boost=10, boost=6.0,
                 q_mode="indep", q_indep_sigma=2.0, temperature=temp,
                 greedy=(kind == 1).astype(np.uint8))
    else:
        raise ValueError(f"no workload {c}")
    if num_reqs is not None and num_reqs < n:
        for key in ("K",):
            b[key] = list(np.asarray(b[key])[:num_reqs])
        if isinstance(b.get("temperature"), np.ndarray):
            b["temperature"] = b["temperature"][:num_reqs]
        if b.get("greedy") is not None:
            b["greedy"] = b["greedy"][:num_reqs]
    name = f"workload{c}"
    if draft_logits:
        if b["q_mode"] not in ("noisy", "indep"):
            raise ValueError(f"workload {c} has no draft distribution")
        b["q_mode"] = "logits"
        b.setdefault("q_noise", 2.0)
        b.pop("q_indep_sigma", None)
        name += "-draft-logits"
    out = make_batch(name=name, data_seed=seed, verify_seed=seed, **b)
    out.meta["workload"] = WORKLOADS[c] + (", draft logits" if draft_logits else "")
    out.meta["index"] = c
    return out
