"""CPU oracle of the verification sampler -- TEST INFRASTRUCTURE ONLY.

Python marshalling for ``sv_oracle.c`` (a plain single-threaded C restatement of the
verification step; see its header for the pages it follows and the readings it takes).
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. The library's product path never uses it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsvoracle.so")
_lib = None

RACE_NONE, RACE_RESIDUAL, RACE_EXCLUDE, RACE_BONUS, RACE_FALLBACK, RACE_TARGET = range(6)


class _Options(ctypes.Structure):
    _fields_ = [("synthetic_rates", ctypes.c_void_p), ("num_synthetic_rates", ctypes.c_int32),
                ("partial_prefill", ctypes.c_void_p), ("frequency_penalty", ctypes.c_void_p),
                ("output_bin_counts", ctypes.c_void_p), ("counts_row", ctypes.c_void_p),
                ("counts_rows", ctypes.c_int32), ("top_k", ctypes.c_void_p),
                ("top_p", ctypes.c_void_p),
                ("row_select_margin", ctypes.c_void_p), ("fp64_gumbel", ctypes.c_int32)]
EBATCH = 1

# Strict IEEE binary32: no contraction of a*b+c into fma (only the explicit fmaf calls
# fuse), no fast-math reassociation.
CFLAGS = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile sv_oracle.c into libsvoracle.so next to it (atomic replace)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    try:
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True, capture_output=True,
                       text=True)
        os.replace(tmp, _LIB_PATH)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp, u32, u64, i32, f32 = (ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int,
                                  ctypes.c_float)
        L.spec_verify_ref_philox.argtypes = [vp, vp, vp]
        L.spec_verify_ref_philox.restype = None
        L.spec_verify_ref_uniform.argtypes = [u64, u32, u32, u32, u32, i32]
        L.spec_verify_ref_uniform.restype = f32
        L.spec_verify_ref_uniform_from_word.argtypes = [u32]
        L.spec_verify_ref_uniform_from_word.restype = f32
        L.spec_verify_ref_exp.argtypes = [f32]
        L.spec_verify_ref_exp.restype = f32
        L.spec_verify_ref_log.argtypes = [f32]
        L.spec_verify_ref_log.restype = f32
        L.spec_verify_ref_run.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, u64, u32, i32, i32, i32,
                                          vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                          ctypes.POINTER(_Options)]
        L.spec_verify_ref_synthetic_rates.argtypes = [ctypes.c_double, i32, vp]
        L.spec_verify_ref_synthetic_rates.restype = i32
        L.spec_verify_ref_run.restype = i32
        L.spec_verify_ref_residual_row.argtypes = [vp, i32, i32, f32, vp, vp, vp, vp, vp]
        L.spec_verify_ref_residual_row.restype = None
        for f in ("spec_verify_ref_exp_n", "spec_verify_ref_log_n"):
            getattr(L, f).argtypes = [vp, vp, ctypes.c_int64]
            getattr(L, f).restype = None
        L.spec_verify_ref_draft_probs.argtypes = [vp, i32, i32, vp, vp, vp, i32, vp]
        L.spec_verify_ref_draft_probs.restype = None
        L.spec_verify_ref_select_row.argtypes = [vp, i32, i32, f32, vp, vp, vp]
        L.spec_verify_ref_select_row.restype = None
        L.spec_verify_ref_shard_stats.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp]
        L.spec_verify_ref_shard_stats.restype = None
        L.spec_verify_ref_shard_race.argtypes = [vp, i32, i32, i32, i32, vp, i32, vp, vp, vp, vp, vp,
                                                 u64, u32, i32, i32, vp]
        L.spec_verify_ref_shard_race.restype = None
        L.spec_verify_ref_shard_finish.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp, vp]
        L.spec_verify_ref_shard_finish.restype = None
        L.spec_verify_ref_race_clocks.argtypes = [u64, u32, u32, i32, vp]
        L.spec_verify_ref_race_clocks.restype = None
        L.spec_verify_ref_race_clocks64.argtypes = [u64, u32, u32, i32, vp]
        L.spec_verify_ref_race_clocks64.restype = None
        L.spec_verify_ref_log64_n.argtypes = [vp, vp, ctypes.c_int64]
        L.spec_verify_ref_log64_n.restype = None
        L.spec_verify_ref_log64.argtypes = [ctypes.c_double]
        L.spec_verify_ref_log64.restype = ctypes.c_double
        L.spec_verify_ref_uniform64.argtypes = [u32, u32]
        L.spec_verify_ref_uniform64.restype = ctypes.c_double
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def philox(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().spec_verify_ref_philox(_p(c), _p(k), _p(out))
    return out


def uniform(seed: int, c0: int, c1: int, c2: int, c3: int, word: int) -> float:
    return lib().spec_verify_ref_uniform(seed, c0, c1, c2, c3, word)


def uniform_from_word(w: int) -> float:
    return lib().spec_verify_ref_uniform_from_word(w)


def exp32(x: float) -> float:
    return lib().spec_verify_ref_exp(x)


def log32(x: float) -> float:
    return lib().spec_verify_ref_log(x)


def exp32_n(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    lib().spec_verify_ref_exp_n(_p(x), _p(out), x.size)
    return out


def log32_n(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    lib().spec_verify_ref_log_n(_p(x), _p(out), x.size)
    return out


def race_clocks(seed: int, j: int, ireq: int, n: int) -> np.ndarray:
    """Race clocks E_v (binary32) of tokens 0..n-1 of (request ireq, position j)."""
    out = np.empty(n, dtype=np.float32)
    lib().spec_verify_ref_race_clocks(seed, j, ireq, n, _p(out))
    return out


def race_clocks64(seed: int, j: int, ireq: int, n: int) -> np.ndarray:
    """Race clocks E_v drawn in binary64 (the fp64 Gumbel option) of tokens 0..n-1."""
    out = np.empty(n, dtype=np.float64)
    lib().spec_verify_ref_race_clocks64(seed, j, ireq, n, _p(out))
    return out


def log64(x: float) -> float:
    return lib().spec_verify_ref_log64(x)


def log64_n(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib().spec_verify_ref_log64_n(_p(x), _p(out), x.size)
    return out


def uniform64(hi: int, lo: int) -> float:
    """52-bit uniform of the binary64 clocks from two Philox words."""
    return lib().spec_verify_ref_uniform64(hi, lo)


def synthetic_rates(mean_length: float, num_spec: int) -> np.ndarray:
    """Minimum-variance per-position rates for a target mean accepted length."""
    out = np.empty(max(num_spec, 0), dtype=np.float32)
    if lib().spec_verify_ref_synthetic_rates(float(mean_length), num_spec, _p(out)) != 0:
        raise ValueError("mean length must lie in [1, num_spec + 1]")
    return out


SHARD_STATS = np.dtype([("ymax", "<f4"), ("amax", "<i4"), ("s", "<f8"), ("ld", "<f4"),
                        ("qd", "<f4")], align=True)
SHARD_RACE = np.dtype([("jstar", "<i4"), ("token", "<i4"), ("res_key", "<f4"), ("res_idx", "<i4"),
                       ("p_key", "<f4"), ("p_idx", "<i4")], align=True)


class ShardOracle:
    """The two-exchange protocol of vocabulary-sharded verification, one rank's side: the
    arrays passed in are this rank's columns [v0, v0 + Vs) of the logits (and of the draft
    probabilities). Exchange records are numpy structured arrays (SHARD_STATS / SHARD_RACE)."""

    def __init__(self, batch, v0: int, shard_vocab: int):
        self.b, self.v0, self.Vs = batch, int(v0), int(shard_vocab)
        lg = np.ascontiguousarray(batch.logits)
        self.logits = np.ascontiguousarray(lg[:, self.v0:self.v0 + self.Vs])
        self.q = None if batch.draft_probs is None else np.ascontiguousarray(
            np.asarray(batch.draft_probs, np.float32)[:, self.v0:self.v0 + self.Vs])
        self.ids = np.ascontiguousarray(batch.draft_ids, np.int32)
        self.cu = np.ascontiguousarray(batch.cu_num_draft, np.int32)
        self.T = np.ascontiguousarray(batch.temperature, np.float32)
        self.g = np.ascontiguousarray(batch.is_greedy, np.uint8)
        self.bf16 = int(batch.logits_dtype == "bf16")

    def stats(self) -> np.ndarray:
        out = np.zeros(self.b.num_rows, SHARD_STATS)
        lib().spec_verify_ref_shard_stats(_p(self.logits), self.bf16, self.Vs, self.v0, _p(self.ids),
                                          _p(self.q), _p(self.cu), _p(self.T), _p(self.g),
                                          self.b.num_reqs, _p(out))
        return out

    def race(self, all_stats: np.ndarray, world: int) -> np.ndarray:
        all_stats = np.ascontiguousarray(all_stats, SHARD_STATS)
        out = np.zeros(self.b.num_reqs, SHARD_RACE)
        lib().spec_verify_ref_shard_race(_p(self.logits), self.bf16, self.Vs, self.v0,
                                         self.b.vocab_size, _p(all_stats), world, _p(self.ids),
                                         _p(self.q), _p(self.cu), _p(self.T), _p(self.g), self.b.seed,
                                         0, self.b.num_reqs, self.b.num_draft_tokens, _p(out))
        return out

    def finish(self, all_races: np.ndarray, world: int, max_spec_len: int):
        all_races = np.ascontiguousarray(all_races, SHARD_RACE)
        n = self.b.num_reqs
        sampled = np.empty((n, max_spec_len + 1), np.int32)
        ns = np.empty(n, np.int32)
        nr = np.empty(n, np.int32)
        lib().spec_verify_ref_shard_finish(_p(all_races), world, _p(self.ids), _p(self.cu), n,
                                           max_spec_len, _p(sampled), _p(ns), _p(nr))
        return sampled, ns, nr


def select_row(x: np.ndarray, top_k: int, top_p: float):
    """(tau, kept mass, top-p margin) of the sampling constraints on one processed row."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    tau = ctypes.c_float()
    Sk = ctypes.c_double()
    margin = ctypes.c_double()
    lib().spec_verify_ref_select_row(_p(x), x.size, int(top_k), float(top_p), ctypes.byref(tau),
                                     ctypes.byref(Sk), ctypes.byref(margin))
    return tau.value, Sk.value, margin.value


def residual_row(logits_row: np.ndarray, bf16: bool, invT: float, q: np.ndarray):
    """t_v = exp(x_v - m), rr_v = fma(-S, q_v, t_v), m, S for one row, as the race uses them."""
    V = logits_row.shape[-1]
    row = np.ascontiguousarray(logits_row)
    q = np.ascontiguousarray(q, dtype=np.float32)
    t = np.empty(V, dtype=np.float32)
    rr = np.empty(V, dtype=np.float32)
    m = ctypes.c_float()
    S = ctypes.c_float()
    lib().spec_verify_ref_residual_row(_p(row), int(bf16), V, invT, _p(q), _p(t), _p(rr),
                                       ctypes.byref(m), ctypes.byref(S))
    return t, rr, m.value, S.value


def draft_probs(draft_logits: np.ndarray, bf16: bool, cu_num_draft, temperature, is_greedy):
    """q = softmax(draft_logits / T_i) per draft row, as the draft-logits mode defines it."""
    dl = np.ascontiguousarray(draft_logits)
    cu = np.ascontiguousarray(cu_num_draft, dtype=np.int32)
    n = cu.shape[0] - 1
    V = dl.shape[-1]
    q = np.zeros((int(cu[-1]), V), dtype=np.float32)
    lib().spec_verify_ref_draft_probs(_p(dl), int(bf16), V, _p(cu),
                                      _p(np.ascontiguousarray(temperature, dtype=np.float32)),
                                      _p(np.ascontiguousarray(is_greedy, dtype=np.uint8)), n, _p(q))
    return q


def run(batch, *, max_spec_len: int | None = None, req_index_base: int = 0, u_override=None,
        seed: int | None = None) -> dict:
    """Run the oracle on a ``workloads.Batch`` (or any object with the same fields).

    Returns sampled, num_sampled, num_rejected, the per-row stats (row_max, row_sumexp,
    row_argmax), the per-position acceptance margins, the per-request race gap and kind,
    j* per request and the status code.
    """
    cu = np.ascontiguousarray(batch.cu_num_draft, dtype=np.int32)
    n = cu.shape[0] - 1
    nd = int(cu[-1])
    R = nd + n
    kmax = batch.max_spec_len if max_spec_len is None else max_spec_len
    V = int(batch.vocab_size)
    logits = np.ascontiguousarray(batch.logits)
    bf16 = batch.logits_dtype == "bf16"
    ids = np.ascontiguousarray(batch.draft_ids, dtype=np.int32)
    q = None if batch.draft_probs is None else np.ascontiguousarray(batch.draft_probs, dtype=np.float32)
    if getattr(batch, "draft_logits", None) is not None:  # draft-logits mode: q from the logits
        if cu.shape[0] - 1 > 0 and (cu[0] != 0 or np.any(np.diff(cu) < 0) or cu[-1] > len(batch.draft_ids)):
            q = np.zeros((len(batch.draft_ids), int(batch.vocab_size)), np.float32)  # never read
        else:
            q = draft_probs(batch.draft_logits, batch.logits_dtype == "bf16", cu,
                            batch.temperature, batch.is_greedy)
    T = np.ascontiguousarray(batch.temperature, dtype=np.float32)
    g = np.ascontiguousarray(batch.is_greedy, dtype=np.uint8)
    out = dict(
        sampled=np.empty((n, kmax + 1), dtype=np.int32),
        num_sampled=np.empty(n, dtype=np.int32),
        num_rejected=np.empty(n, dtype=np.int32),
        row_max=np.empty(R, dtype=np.float32),
        row_sumexp=np.empty(R, dtype=np.float32),
        row_argmax=np.empty(R, dtype=np.int32),
        accept_margin=np.empty(max(nd, 1), dtype=np.float64),
        race_gap=np.empty(max(n, 1), dtype=np.float64),
        race_kind=np.empty(max(n, 1), dtype=np.int32),
        jstar=np.empty(max(n, 1), dtype=np.int32),
    )
    uo = None if u_override is None else np.ascontiguousarray(u_override, dtype=np.float32)
    s = batch.seed if seed is None else seed
    opts = _Options()
    rates = getattr(batch, "synthetic_rates", None)
    if rates is not None:
        rates = np.ascontiguousarray(rates, dtype=np.float32)
        opts.synthetic_rates = rates.ctypes.data
        opts.num_synthetic_rates = rates.size
    partial = getattr(batch, "partial_prefill", None)
    if partial is not None:
        partial = np.ascontiguousarray(partial, dtype=np.uint8)
        opts.partial_prefill = partial.ctypes.data
    keep = []  # arrays whose addresses the options hold

    def _opt(name, dtype):
        a = getattr(batch, name, None)
        if a is None:
            return None
        a = np.ascontiguousarray(a, dtype=dtype)
        keep.append(a)
        return a.ctypes.data

    opts.frequency_penalty = _opt("frequency_penalty", np.float32)
    opts.output_bin_counts = _opt("output_bin_counts", np.int32)
    opts.counts_row = _opt("counts_row", np.int32)
    if getattr(batch, "output_bin_counts", None) is not None:
        opts.counts_rows = int(np.asarray(batch.output_bin_counts).shape[0])
    opts.top_k = _opt("top_k", np.int32)
    opts.top_p = _opt("top_p", np.float32)
    opts.fp64_gumbel = int(bool(getattr(batch, "fp64_gumbel", False)))
    out["row_select_margin"] = np.empty(max(R, 1), dtype=np.float64)
    opts.row_select_margin = out["row_select_margin"].ctypes.data
    rc = lib().spec_verify_ref_run(
        _p(logits), int(bf16), V, _p(ids), _p(q), _p(cu), _p(T), _p(g), s, req_index_base, n, nd,
        kmax, _p(out["sampled"]), _p(out["num_sampled"]), _p(out["num_rejected"]), _p(out["row_max"]),
        _p(out["row_sumexp"]), _p(out["row_argmax"]), _p(out["accept_margin"]), _p(out["race_gap"]),
        _p(out["race_kind"]), _p(out["jstar"]), _p(uo), ctypes.byref(opts))
    out["accept_margin"] = out["accept_margin"][:nd]
    out["row_select_margin"] = out["row_select_margin"][:R]
    for k in ("race_gap", "race_kind", "jstar"):
        out[k] = out[k][:n]
    out["status"] = rc
    return out
