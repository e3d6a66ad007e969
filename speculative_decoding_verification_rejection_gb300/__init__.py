"""GB300-native speculative-decoding verification sampler.

Python binding of the C ABI in ``include/spec_verify.h`` (``libspecverify.so``, built in-tree
for sm_103a by :func:`build`). This module only marshals arguments: every step of the
verification runs in the library's CUDA kernels. PyTorch tensors are accepted for device
memory and streams; raw integer pointers work as well.

The same names as the C ABI are exported (``spec_verify_init``, ``spec_verify_run``, ...),
plus :class:`SpecVerify`, a small owner of a context.
"""
from __future__ import annotations

import ctypes
import os
import re
import subprocess
import tempfile

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_INCLUDE = os.path.join(_ROOT, "include")
_HEADER = os.path.join(_INCLUDE, "spec_verify.h")
_SOURCES = [os.path.join(_PKG, "csrc", "spec_verify.cu"), os.path.join(_PKG, "csrc", "sv_device.cuh")]
# SPEC_VERIFY_DEBUG_BOUNDS=1 in the environment selects the checked build (-DSV_DEBUG_BOUNDS): every
# global load and store of the kernels is checked against the call's arrays, and an access
# outside them is skipped and reported as SV_ERR_BOUNDS in the error word. For tests only.
DEBUG_BOUNDS = os.environ.get("SPEC_VERIFY_DEBUG_BOUNDS", "0") not in ("", "0")
RELEASE_LIB_PATH = os.path.join(_PKG, "libspecverify.so")
DEBUG_LIB_PATH = os.path.join(_PKG, "libspecverify_debug.so")
LIB_PATH = DEBUG_LIB_PATH if DEBUG_BOUNDS else RELEASE_LIB_PATH

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-shared", "-Xcompiler", "-fPIC", "-I" + _INCLUDE]

SV_OK, SV_EINVAL, SV_ECAPACITY, SV_EDTYPE, SV_ECUDA, SV_EDEVICE = 0, -1, -2, -3, -4, -5
SV_F32, SV_BF16 = 0, 1
SV_DRAFT_PROBS, SV_DRAFT_LOGITS = 1, 2
SV_MAX_SYNTHETIC = 64


class Batch(ctypes.Structure):
    """spec_verify_batch of include/spec_verify.h."""
    _fields_ = [("logits", ctypes.c_void_p), ("draft_ids", ctypes.c_void_p),
                ("draft_probs", ctypes.c_void_p), ("draft_logits", ctypes.c_void_p),
                ("cu_num_draft", ctypes.c_void_p), ("temperature", ctypes.c_void_p),
                ("is_greedy", ctypes.c_void_p), ("partial_prefill", ctypes.c_void_p),
                ("frequency_penalty", ctypes.c_void_p), ("output_bin_counts", ctypes.c_void_p),
                ("counts_row", ctypes.c_void_p), ("top_k", ctypes.c_void_p),
                ("top_p", ctypes.c_void_p),
                ("seed", ctypes.c_uint64), ("req_index_base", ctypes.c_uint32),
                ("num_reqs", ctypes.c_int32), ("num_draft_tokens", ctypes.c_int32),
                ("max_spec_len_this_batch", ctypes.c_int32), ("counts_rows", ctypes.c_int32),
                ("fp64_gumbel", ctypes.c_int32)]


class Outputs(ctypes.Structure):
    """spec_verify_outputs of include/spec_verify.h."""
    _fields_ = [("sampled", ctypes.c_void_p), ("num_sampled", ctypes.c_void_p),
                ("num_rejected", ctypes.c_void_p), ("row_max", ctypes.c_void_p),
                ("row_sumexp", ctypes.c_void_p), ("row_argmax", ctypes.c_void_p)]
SV_ERR_BATCH, SV_ERR_COUNTS, SV_ERR_BOUNDS, SV_ERR_SELECT = 1, 2, 4, 8
KERNELS = ("stats", "verify", "select")  # profiling slots (select: top-k / top-p calls)

_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = _status_string(status)
        super().__init__(f"{what}: {msg} ({status})")
        self.status = status


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(path: str | None = None) -> bool:
    path = path or LIB_PATH
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(s) > t for s in _SOURCES + [_HEADER])


def build(force: bool = False, verbose: bool = False, debug: bool | None = None) -> str:
    """Compile libspecverify.so (or, with debug=True, the checked libspecverify_debug.so) for
    sm_103a next to this file (atomic replace). debug=None: the build this process loads."""
    debug = DEBUG_BOUNDS if debug is None else debug
    path = DEBUG_LIB_PATH if debug else RELEASE_LIB_PATH
    if not force and not _stale(path):
        return path
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_PKG)
    os.close(fd)
    cmd = [_nvcc(), *NVCC_FLAGS, *(["-DSV_DEBUG_BOUNDS"] if debug else []), "-o", tmp, _SOURCES[0]]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stderr[-4000:])
        if verbose:
            print(r.stderr)
        os.replace(tmp, path)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return path


def build_all(force: bool = False) -> None:
    """Both builds (the library and its checked debug variant), compiled in parallel."""
    import threading

    errors = []

    def one(debug):
        try:
            build(force=force, debug=debug)
        except Exception as e:  # noqa: BLE001 - re-raised below
            errors.append(e)

    threads = [threading.Thread(target=one, args=(d,)) for d in (False, True)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        raise errors[0]


def declared_symbols() -> list[str]:
    """Names of the functions include/spec_verify.h declares."""
    with open(_HEADER, encoding="utf-8") as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(spec_verify_\w+)\s*\(", text, re.M)))


def lib():
    """The loaded C library (ctypes), built first if missing. Raises if it cannot be built or
    loaded: there is no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    if _stale():
        # a library older than its sources is never loaded: a failed rebuild raises, so that a
        # compile error cannot leave the previous binary running (and measured) in its place
        try:
            build()
        except (OSError, RuntimeError) as e:
            raise RuntimeError("libspecverify.so is out of date and could not be rebuilt: "
                               + str(e)) from e
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u32, u64, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64
    L.spec_verify_init.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32]
    L.spec_verify_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, u64, u32, i32, i32, i32, vp, vp, vp,
                                  vp, vp, vp, vp]
    L.spec_verify_run_draft_logits.argtypes = list(L.spec_verify_run.argtypes)
    L.spec_verify_run_batch.argtypes = [vp, ctypes.POINTER(Batch), ctypes.POINTER(Outputs), vp]
    L.spec_verify_set_synthetic.argtypes = [vp, vp, i32]
    L.spec_verify_shard_stats.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp]
    L.spec_verify_shard_race.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, vp, vp, vp, u64, u32,
                                         i32, i32, i32, vp, vp]
    L.spec_verify_shard_finish.argtypes = [vp, vp, i32, vp, vp, i32, i32, vp, vp, vp, vp]
    L.spec_verify_synthetic_rates.argtypes = [ctypes.c_double, i32, vp]
    L.spec_verify_run_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, u64, u32, i32, i32, i32, vp, vp,
                                       vp, vp]
    L.spec_verify_run_noalloc.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, u64, u32, i32, i32,
                                          i32, vp, vp, vp, vp, vp, vp, vp]
    L.spec_verify_noalloc_last_error.argtypes = [ctypes.POINTER(u32)]
    L.spec_verify_reserve_host_io.argtypes = [vp]
    L.spec_verify_last_error.argtypes = [vp, ctypes.POINTER(u32)]
    L.spec_verify_set_profiling.argtypes = [vp, i32]
    L.spec_verify_get_profile.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]
    L.spec_verify_set_chunks.argtypes = [vp, i32]
    L.spec_verify_launches_per_run.argtypes = []
    L.spec_verify_free.argtypes = [vp]
    L.spec_verify_free.restype = None
    L.spec_verify_status_string.argtypes = [i32]
    L.spec_verify_status_string.restype = ctypes.c_char_p
    for f in ("spec_verify_init", "spec_verify_run", "spec_verify_run_draft_logits",
              "spec_verify_run_batch", "spec_verify_set_synthetic", "spec_verify_synthetic_rates",
              "spec_verify_shard_stats", "spec_verify_shard_race", "spec_verify_shard_finish",
              "spec_verify_run_host", "spec_verify_run_noalloc", "spec_verify_noalloc_last_error",
              "spec_verify_reserve_host_io", "spec_verify_last_error", "spec_verify_set_profiling",
              "spec_verify_get_profile", "spec_verify_set_chunks", "spec_verify_launches_per_run"):
        getattr(L, f).restype = i32
    _lib = L
    return L


def _status_string(status: int) -> str:
    try:
        return lib().spec_verify_status_string(status).decode()
    except Exception:  # noqa: BLE001 - only for messages
        return "status"


def _check(status: int, what: str) -> None:
    if status != SV_OK:
        raise SpecVerifyError(status, what)


def _ptr(x):
    """Device or host address of a tensor / array / int (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensors must be contiguous")
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- thin wrappers with the C names --------------------------------------------------------

def spec_verify_init(max_num_reqs: int, max_spec_len: int, vocab_size: int, logits_dtype: int,
                     draft_input: int, device: int) -> int:
    ctx = ctypes.c_void_p()
    _check(lib().spec_verify_init(ctypes.byref(ctx), max_num_reqs, max_spec_len, vocab_size,
                                  logits_dtype, draft_input, device), "spec_verify_init")
    return ctx.value


def spec_verify_run(ctx, logits, draft_ids, draft_probs, cu_num_draft, temperature, is_greedy,
                    seed, req_index_base, num_reqs, num_draft_tokens, max_spec_len_this_batch,
                    sampled, num_sampled, num_rejected, opt_row_max=None, opt_row_sumexp=None,
                    opt_row_argmax=None, cuda_stream=None) -> None:
    _check(lib().spec_verify_run(ctx, _ptr(logits), _ptr(draft_ids), _ptr(draft_probs),
                                 _ptr(cu_num_draft), _ptr(temperature), _ptr(is_greedy), seed,
                                 req_index_base, num_reqs, num_draft_tokens,
                                 max_spec_len_this_batch, _ptr(sampled), _ptr(num_sampled),
                                 _ptr(num_rejected), _ptr(opt_row_max), _ptr(opt_row_sumexp),
                                 _ptr(opt_row_argmax), _stream_handle(cuda_stream)),
           "spec_verify_run")


def spec_verify_run_draft_logits(ctx, logits, draft_ids, draft_logits, cu_num_draft, temperature,
                                 is_greedy, seed, req_index_base, num_reqs, num_draft_tokens,
                                 max_spec_len_this_batch, sampled, num_sampled, num_rejected,
                                 opt_row_max=None, opt_row_sumexp=None, opt_row_argmax=None,
                                 cuda_stream=None) -> None:
    _check(lib().spec_verify_run_draft_logits(
        ctx, _ptr(logits), _ptr(draft_ids), _ptr(draft_logits), _ptr(cu_num_draft),
        _ptr(temperature), _ptr(is_greedy), seed, req_index_base, num_reqs, num_draft_tokens,
        max_spec_len_this_batch, _ptr(sampled), _ptr(num_sampled), _ptr(num_rejected),
        _ptr(opt_row_max), _ptr(opt_row_sumexp), _ptr(opt_row_argmax),
        _stream_handle(cuda_stream)), "spec_verify_run_draft_logits")


def spec_verify_run_batch(ctx, batch: Batch, out: Outputs, cuda_stream=None) -> None:
    _check(lib().spec_verify_run_batch(ctx, ctypes.byref(batch), ctypes.byref(out),
                                       _stream_handle(cuda_stream)), "spec_verify_run_batch")


def spec_verify_set_synthetic(ctx, rates) -> None:
    """rates: host sequence of unconditional per-position acceptance rates ([] = off)."""
    import numpy as np
    r = np.ascontiguousarray(np.asarray(rates, dtype=np.float32).reshape(-1))
    _check(lib().spec_verify_set_synthetic(ctx, r.ctypes.data if r.size else None, r.size),
           "spec_verify_set_synthetic")


def spec_verify_synthetic_rates(mean_length: float, num_spec: int):
    """Minimum-variance per-position rates for a target mean accepted length (numpy float32)."""
    import numpy as np
    out = np.zeros(max(num_spec, 0), dtype=np.float32)
    _check(lib().spec_verify_synthetic_rates(float(mean_length), num_spec,
                                             out.ctypes.data if out.size else None),
           "spec_verify_synthetic_rates")
    return out


SHARD_RECORD_BYTES = 24  # spec_verify_shard_stat and spec_verify_shard_key


def spec_verify_shard_stats(ctx, logits_shard, v0, draft_ids, draft_probs_shard, cu_num_draft,
                            temperature, is_greedy, num_reqs, num_draft_tokens,
                            max_spec_len_this_batch, out, cuda_stream=None) -> None:
    _check(lib().spec_verify_shard_stats(ctx, _ptr(logits_shard), v0, _ptr(draft_ids),
                                         _ptr(draft_probs_shard), _ptr(cu_num_draft),
                                         _ptr(temperature), _ptr(is_greedy), num_reqs,
                                         num_draft_tokens, max_spec_len_this_batch, _ptr(out),
                                         _stream_handle(cuda_stream)), "spec_verify_shard_stats")


def spec_verify_shard_race(ctx, logits_shard, v0, vocab_size, all_stats, world, draft_ids,
                           draft_probs_shard, cu_num_draft, temperature, is_greedy, seed,
                           req_index_base, num_reqs, num_draft_tokens, max_spec_len_this_batch,
                           out, cuda_stream=None) -> None:
    _check(lib().spec_verify_shard_race(ctx, _ptr(logits_shard), v0, vocab_size, _ptr(all_stats),
                                        world, _ptr(draft_ids), _ptr(draft_probs_shard),
                                        _ptr(cu_num_draft), _ptr(temperature), _ptr(is_greedy),
                                        seed, req_index_base, num_reqs, num_draft_tokens,
                                        max_spec_len_this_batch, _ptr(out),
                                        _stream_handle(cuda_stream)), "spec_verify_shard_race")


def spec_verify_shard_finish(ctx, all_races, world, draft_ids, cu_num_draft, num_reqs,
                             max_spec_len_this_batch, sampled, num_sampled, num_rejected,
                             cuda_stream=None) -> None:
    _check(lib().spec_verify_shard_finish(ctx, _ptr(all_races), world, _ptr(draft_ids),
                                          _ptr(cu_num_draft), num_reqs, max_spec_len_this_batch,
                                          _ptr(sampled), _ptr(num_sampled), _ptr(num_rejected),
                                          _stream_handle(cuda_stream)), "spec_verify_shard_finish")


def spec_verify_run_host(ctx, logits, draft_ids, draft_probs, cu_num_draft, temperature,
                         is_greedy, seed, req_index_base, num_reqs, num_draft_tokens,
                         max_spec_len_this_batch, sampled, num_sampled, num_rejected,
                         cuda_stream=None) -> None:
    _check(lib().spec_verify_run_host(ctx, _ptr(logits), _ptr(draft_ids), _ptr(draft_probs),
                                      _ptr(cu_num_draft), _ptr(temperature), _ptr(is_greedy), seed,
                                      req_index_base, num_reqs, num_draft_tokens,
                                      max_spec_len_this_batch, _ptr(sampled), _ptr(num_sampled),
                                      _ptr(num_rejected), _stream_handle(cuda_stream)),
           "spec_verify_run_host")


def spec_verify_run_noalloc(logits, logits_dtype, vocab_size, draft_ids, draft_probs,
                            cu_num_draft, temperature, is_greedy, seed, req_index_base, num_reqs,
                            num_draft_tokens, max_spec_len_this_batch, sampled, num_sampled,
                            num_rejected, opt_row_max=None, opt_row_sumexp=None,
                            opt_row_argmax=None, cuda_stream=None) -> None:
    """Verification that allocates nothing (scratch in a static device array of the library,
    limits SV_NOALLOC_MAX_*), for callers that cannot allocate device memory. Runs on the
    current device; overlapping calls on one device race and must be serialised."""
    _check(lib().spec_verify_run_noalloc(_ptr(logits), _dtype_code(logits_dtype)
                                         if isinstance(logits_dtype, str) else logits_dtype,
                                         vocab_size, _ptr(draft_ids), _ptr(draft_probs),
                                         _ptr(cu_num_draft), _ptr(temperature), _ptr(is_greedy),
                                         seed, req_index_base, num_reqs, num_draft_tokens,
                                         max_spec_len_this_batch, _ptr(sampled), _ptr(num_sampled),
                                         _ptr(num_rejected), _ptr(opt_row_max),
                                         _ptr(opt_row_sumexp), _ptr(opt_row_argmax),
                                         _stream_handle(cuda_stream)),
           "spec_verify_run_noalloc")


def spec_verify_noalloc_last_error() -> int:
    """Read and clear the error word of spec_verify_run_noalloc on the current device (waits
    for the device)."""
    w = ctypes.c_uint32()
    _check(lib().spec_verify_noalloc_last_error(ctypes.byref(w)), "spec_verify_noalloc_last_error")
    return w.value


def spec_verify_reserve_host_io(ctx) -> None:
    _check(lib().spec_verify_reserve_host_io(ctx), "spec_verify_reserve_host_io")


def spec_verify_last_error(ctx) -> int:
    w = ctypes.c_uint32()
    _check(lib().spec_verify_last_error(ctx, ctypes.byref(w)), "spec_verify_last_error")
    return w.value


def spec_verify_set_profiling(ctx, enable: bool) -> None:
    _check(lib().spec_verify_set_profiling(ctx, int(enable)), "spec_verify_set_profiling")


def spec_verify_get_profile(ctx):
    ms = (ctypes.c_double * len(KERNELS))()
    calls = ctypes.c_int64()
    _check(lib().spec_verify_get_profile(ctx, ms, ctypes.byref(calls)), "spec_verify_get_profile")
    return dict(zip(KERNELS, list(ms))), calls.value


def spec_verify_set_chunks(ctx, stats_chunk: int = 0) -> None:
    _check(lib().spec_verify_set_chunks(ctx, stats_chunk), "spec_verify_set_chunks")


def spec_verify_launches_per_run() -> int:
    return lib().spec_verify_launches_per_run()


def spec_verify_free(ctx) -> None:
    if ctx:
        lib().spec_verify_free(ctx)


def spec_verify_status_string(status: int) -> str:
    return _status_string(status)


# ---- convenience owner ---------------------------------------------------------------------

def _dtype_code(logits_dtype) -> int:
    s = str(logits_dtype).lower()
    if "bf16" in s or "bfloat16" in s:
        return SV_BF16
    if "f32" in s or "float32" in s or s in ("float", "torch.float"):
        return SV_F32
    raise ValueError(f"unsupported logits dtype {logits_dtype}")


class SpecVerify:
    """Owns one context. Tensors passed to :meth:`run` must live on the context's device."""

    def __init__(self, max_num_reqs: int, max_spec_len: int, vocab_size: int, logits_dtype="bf16",
                 has_draft_probs: bool = True, device: int = 0, *, draft_logits: bool = False):
        self.max_num_reqs, self.max_spec_len, self.vocab_size = max_num_reqs, max_spec_len, vocab_size
        self.dtype_code = _dtype_code(logits_dtype)
        self.device = device
        draft_input = (SV_DRAFT_PROBS if has_draft_probs else 0) | (SV_DRAFT_LOGITS if draft_logits else 0)
        self.ctx = spec_verify_init(max_num_reqs, max_spec_len, vocab_size, self.dtype_code,
                                    draft_input, device)

    def run(self, logits, draft_ids, draft_probs, cu_num_draft, temperature, is_greedy, seed: int,
            *, req_index_base: int = 0, max_spec_len: int | None = None, out=None,
            row_stats: bool = False, stream=None, draft_logits=None, partial_prefill=None,
            frequency_penalty=None, output_bin_counts=None, counts_row=None, top_k=None,
            top_p=None, stats_out=None, fp64_gumbel: bool = False):
        """Verify a batch held in device tensors. Returns (sampled, num_sampled, num_rejected)
        and, with row_stats=True, also (row_max, row_sumexp, row_argmax).

        draft_logits ([num_draft_tokens, vocab_size], the logits' dtype) replaces draft_probs:
        q is then computed inside the call (context created with draft_logits=True).
        partial_prefill ([num_reqs] uint8): requests still in a chunked prefill, which report
        no token. frequency_penalty ([num_reqs] float32) with output_bin_counts ([rows, V]
        int32) and counts_row ([num_reqs] int32, optional): the frequency penalty. top_k
        ([num_reqs] int32), top_p ([num_reqs] float32): sampling constraints. Any of these
        goes through spec_verify_run_batch. out / stats_out: caller-provided output tensors
        (sampled, num_sampled, num_rejected) / (row_max, row_sumexp, row_argmax).
        fp64_gumbel=True draws the race noise in binary64 (the fp64 Gumbel option)."""
        import torch
        num_reqs = cu_num_draft.numel() - 1
        nd = draft_ids.numel()
        kmax = self.max_spec_len if max_spec_len is None else max_spec_len
        if logits.dim() != 2 or logits.shape[0] != nd + num_reqs or logits.shape[1] != self.vocab_size:
            raise ValueError("logits must be [num_draft_tokens + num_reqs, vocab_size]")
        if draft_logits is not None:
            if draft_probs is not None:
                raise ValueError("give draft_probs or draft_logits, not both")
            if (draft_logits.dim() != 2 or draft_logits.shape[0] != nd
                    or draft_logits.shape[1] != self.vocab_size or draft_logits.dtype != logits.dtype):
                raise ValueError("draft_logits must be [num_draft_tokens, vocab_size] of the logits' dtype")
        dev = logits.device
        if out is None:
            out = (torch.empty((num_reqs, kmax + 1), dtype=torch.int32, device=dev),
                   torch.empty(num_reqs, dtype=torch.int32, device=dev),
                   torch.empty(num_reqs, dtype=torch.int32, device=dev))
        stats = (None, None, None)
        if row_stats and stats_out is not None:
            stats = tuple(stats_out)
        elif row_stats:
            R = nd + num_reqs
            stats = (torch.empty(R, dtype=torch.float32, device=dev),
                     torch.empty(R, dtype=torch.float32, device=dev),
                     torch.empty(R, dtype=torch.int32, device=dev))
        extras = (partial_prefill, frequency_penalty, output_bin_counts, counts_row, top_k, top_p)
        if any(x is not None for x in extras) or fp64_gumbel:
            if output_bin_counts is not None and (output_bin_counts.dim() != 2
                                                  or output_bin_counts.shape[1] != self.vocab_size):
                raise ValueError("output_bin_counts must be [rows, vocab_size]")
            b = Batch(_ptr(logits), _ptr(draft_ids), _ptr(draft_probs), _ptr(draft_logits),
                      _ptr(cu_num_draft), _ptr(temperature), _ptr(is_greedy),
                      _ptr(partial_prefill), _ptr(frequency_penalty), _ptr(output_bin_counts),
                      _ptr(counts_row), _ptr(top_k), _ptr(top_p), seed, req_index_base,
                      num_reqs, nd, kmax,
                      output_bin_counts.shape[0] if output_bin_counts is not None else 0,
                      int(bool(fp64_gumbel)))
            o = Outputs(*(_ptr(t) for t in (*out, *stats)))
            spec_verify_run_batch(self.ctx, b, o, cuda_stream=stream)
        elif draft_logits is not None:
            spec_verify_run_draft_logits(self.ctx, logits, draft_ids, draft_logits, cu_num_draft,
                                         temperature, is_greedy, seed, req_index_base, num_reqs,
                                         nd, kmax, *out, *stats, cuda_stream=stream)
        else:
            spec_verify_run(self.ctx, logits, draft_ids, draft_probs, cu_num_draft, temperature,
                            is_greedy, seed, req_index_base, num_reqs, nd, kmax, *out, *stats,
                            cuda_stream=stream)
        return (*out, *stats) if row_stats else out

    def reserve_host_io(self) -> None:
        spec_verify_reserve_host_io(self.ctx)

    def run_host(self, logits, draft_ids, draft_probs, cu_num_draft, temperature, is_greedy,
                 seed: int, sampled, num_sampled, num_rejected, *, req_index_base: int = 0,
                 max_spec_len: int | None = None, stream=None) -> None:
        """Verify a batch held in host memory (numpy arrays or CPU tensors; pinned memory
        gives asynchronous copies, and pinned draft_probs is read in place by the kernels);
        outputs are written to the host arrays given."""
        num_reqs = len(cu_num_draft) - 1
        nd = len(draft_ids)
        kmax = self.max_spec_len if max_spec_len is None else max_spec_len
        spec_verify_run_host(self.ctx, logits, draft_ids, draft_probs, cu_num_draft, temperature,
                             is_greedy, seed, req_index_base, num_reqs, nd, kmax, sampled,
                             num_sampled, num_rejected, cuda_stream=stream)

    def last_error(self) -> int:
        return spec_verify_last_error(self.ctx)

    def set_profiling(self, enable: bool) -> None:
        spec_verify_set_profiling(self.ctx, enable)

    def get_profile(self):
        return spec_verify_get_profile(self.ctx)

    def set_synthetic(self, rates) -> None:
        """Synthetic acceptance with these unconditional per-position rates ([] = off)."""
        spec_verify_set_synthetic(self.ctx, rates)

    def set_synthetic_length(self, mean_length: float, num_spec: int | None = None) -> None:
        """Synthetic acceptance with the minimum-variance rates of a target mean length."""
        n = self.max_spec_len if num_spec is None else num_spec
        spec_verify_set_synthetic(self.ctx, spec_verify_synthetic_rates(mean_length, n))

    def set_chunks(self, stats_chunk: int = 0) -> None:
        spec_verify_set_chunks(self.ctx, stats_chunk)

    def close(self) -> None:
        if self.ctx:
            spec_verify_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass
