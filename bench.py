#!/usr/bin/env python
"""Benchmark of the GB300 speculative-decoding verification sampler.

One step = one call of the verification step (both kernels: row statistics, then verify =
acceptance + race + emit) on one batch of the bandwidth workload: 256 requests x (K=5 draft positions + 1 bonus) = 1536 logit rows of a
151936-token vocabulary in bf16, fp32 draft distributions for the 1280 draft positions
(1245 MB of inputs, larger than the 129 MB L2, so no flush is needed between steps).

Prints one JSON line (rank 0). Metric: verified draft positions per second, whole job.
  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload 0..4]
                  [--draft-logits]
--draft-logits measures the draft-logits input mode on the same recipe: the draft model's bf16
logits replace the fp32 distributions, and q = softmax(draft logits / T) is computed in the call.
--synthetic-length L measures synthetic acceptance (per-position rates of mean length L).
--top-p P, --top-k K and --frequency-penalty measure the logits processors on the same recipe.
--vocab-shards N measures the vocabulary-sharded protocol (N ranks' calls in turn on one GPU).
Under torchrun (N > 1) every rank verifies its own batch (weak scaling, no collective on the
data path); the step time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec"
UNIT = "positions/s"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCE = os.path.join(ROOT, "speculative_decoding_verification_rejection_gb300", "csrc",
                             "spec_verify.cu")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", type=int, default=3)
    p.add_argument("--num-reqs", type=int, default=None,
                   help="only the first N requests of the workload (bounded cases for profiling)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--profile-steps", type=int, default=500)
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="CPU work of the oracle baseline sample (seconds)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--draft-logits", action="store_true",
                   help="draft logits instead of draft probabilities (q computed in the call)")
    p.add_argument("--synthetic-length", type=float, default=None,
                   help="synthetic acceptance with the minimum-variance rates of this mean length")
    p.add_argument("--top-p", type=float, default=None, help="top-p of every request")
    p.add_argument("--top-k", type=int, default=None, help="top-k of every request")
    p.add_argument("--frequency-penalty", action="store_true",
                   help="a frequency penalty with seeded output-token counts per request")
    p.add_argument("--stats-chunk", type=int, default=0,
                   help="elements per statistics CTA (0: the library's automatic split)")
    p.add_argument("--fp64-gumbel", action="store_true",
                   help="race noise drawn in binary64 (the fp64 Gumbel option)")
    p.add_argument("--vocab-shards", type=int, default=1,
                   help="vocabulary-sharded verification with N shards, their calls emulated in "
                        "turn on one GPU (the exchange a concatenation)")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def load_workload(args, num_reqs=None):
    """The bench's batch: workload recipe, draft-logits and synthetic options applied."""
    import workloads

    b = workloads.workload(args.workload, num_reqs=num_reqs, draft_logits=args.draft_logits)
    if args.synthetic_length is not None:
        import speculative_decoding_verification_rejection_gb300 as sv
        b.synthetic_rates = sv.spec_verify_synthetic_rates(args.synthetic_length, b.max_spec_len)
    import numpy as np
    if args.top_p is not None:
        b.top_p = np.full(b.num_reqs, args.top_p, np.float32)
    if args.top_k is not None:
        b.top_k = np.full(b.num_reqs, args.top_k, np.int32)
    if args.frequency_penalty:
        workloads.add_penalty(b, args.workload)
    b.fp64_gumbel = bool(args.fp64_gumbel)
    return b


def workload_config(b):
    return {
        "workload": f"{b.num_reqs} requests, K={b.max_spec_len} draft tokens + 1 bonus each, "
                    f"V={b.vocab_size}, {b.logits_dtype} logits ({b.meta.get('workload', '')})",
        "num_reqs": b.num_reqs,
        "draft_positions": b.num_draft_tokens,
        "logit_rows": b.num_rows,
        "vocab": b.vocab_size,
        "logits_dtype": b.logits_dtype,
        "draft_probs": "fp32" if b.draft_probs is not None else "none",
        "draft_logits": b.logits_dtype if b.draft_logits is not None else "none",
        "synthetic_rates": None if b.synthetic_rates is None else [float(x) for x in b.synthetic_rates],
        "top_p": None if b.top_p is None else float(b.top_p[0]),
        "top_k": None if b.top_k is None else int(b.top_k[0]),
        "frequency_penalty": b.frequency_penalty is not None,
        "fp64_gumbel": bool(b.fp64_gumbel),
        "input_mb": round((b.logits.nbytes + (b.draft_probs.nbytes if b.draft_probs is not None else 0)
                           + (b.draft_logits.nbytes if b.draft_logits is not None else 0)) / 1e6, 2),
    }


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    def __init__(self, gpu_index: str):
        self.samples = []  # (t, sm, max, power, reasons_active dict)
        self.proc = None
        self.err = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", gpu_index], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError as e:
            self.err = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                pw = float(parts[3])
            except ValueError:
                pw = None
            act = {r: parts[5 + k].lower().startswith("active") for k, r in enumerate(REASONS)}
            self.samples.append((time.perf_counter(), sm, mx, pw, act))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": f"nvidia-smi unavailable: {self.err}"}
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "samples inside the timed region"
        if not win:  # timed region shorter than the sampling period: nearest samples
            win = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            note = "timed region shorter than the 50 ms sampling period: nearest samples"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}
        sm = sorted(s[1] for s in win)
        reasons = sorted({r for s in win for r, a in s[4].items() if a})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(s[2] for s in win), "reasons": reasons,
                "samples": len(win), "power_w_max": max((s[3] or 0) for s in win), "note": note}


def gpu_index_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ---------------------------------------------------------------------------------------------
# roofline helpers
# ---------------------------------------------------------------------------------------------
def measured_peak_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def recorded_traffic(summary: str):
    """DRAM bytes per launch of the stats kernel from the committed ncu summary, if the kernel
    source has not changed since it was taken (source hash recorded in the summary)."""
    import hashlib
    try:
        with open(os.path.join(PROFILE_DIR, summary), encoding="utf-8") as f:
            text = f.read()
        with open(KERNEL_SOURCE, "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None, "no ncu summary"
    fields = dict(l.split(":", 1) for l in text.splitlines() if l.startswith(("traffic_bytes_per_launch:", "kernel_source_sha256_16:")))
    if fields.get("kernel_source_sha256_16", "").strip() != digest:
        return None, "kernel changed since the ncu capture"
    try:
        return int(fields["traffic_bytes_per_launch"].strip()), "ncu dram__bytes_read.sum + dram__bytes_write.sum"
    except (KeyError, ValueError):
        return None, "no traffic line"


# ---------------------------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------------------------
def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo", encoding="utf-8") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def request_slice(b, lo: int, hi: int):
    """Requests [lo, hi) of a batch as a batch of their own (verified with req_index_base = lo,
    which keys every draw as in the whole batch)."""
    import numpy as np
    import workloads

    cu = b.cu_num_draft
    r0, r1 = int(cu[lo]) + lo, int(cu[hi]) + hi
    q0, q1 = int(cu[lo]), int(cu[hi])
    return workloads.Batch(
        name=f"{b.name}[{lo}:{hi}]", logits=b.logits[r0:r1], logits_dtype=b.logits_dtype,
        vocab_size=b.vocab_size, draft_ids=b.draft_ids[q0:q1],
        draft_probs=None if b.draft_probs is None else b.draft_probs[q0:q1],
        cu_num_draft=(cu[lo:hi + 1] - cu[lo]).astype(np.int32),
        temperature=b.temperature[lo:hi], is_greedy=b.is_greedy[lo:hi], seed=b.seed,
        draft_logits=None if b.draft_logits is None else b.draft_logits[q0:q1],
        synthetic_rates=b.synthetic_rates,
        frequency_penalty=None if b.frequency_penalty is None else b.frequency_penalty[lo:hi],
        output_bin_counts=b.output_bin_counts,
        counts_row=(np.arange(lo, hi, dtype=np.int32) if b.counts_row is None else b.counts_row[lo:hi])
        if b.frequency_penalty is not None else None,
        top_k=None if b.top_k is None else b.top_k[lo:hi],
        top_p=None if b.top_p is None else b.top_p[lo:hi], fp64_gumbel=b.fp64_gumbel)


def time_oracle(args, seconds: float):
    """Time the oracle (as it stands: single-threaded C) on the first requests of the workload,
    enough of them for about `seconds` of CPU work on one core: once on one thread, then split
    by requests over every host core (one thread per core, each running the unchanged oracle
    on its own requests; ctypes releases the interpreter lock during the call)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    one = load_workload(args, num_reqs=2)
    t = time.perf_counter()
    oracle.run(one)
    per_req = max((time.perf_counter() - t) / one.num_reqs, 1e-4)
    n = max(2, int(seconds / per_req))
    b = load_workload(args, num_reqs=n)
    t = time.perf_counter()
    oracle.run(b)
    dt = time.perf_counter() - t
    cores = host_cores()
    n = b.num_reqs
    parts = [(n * k // cores, n * (k + 1) // cores) for k in range(cores)]
    subs = [(lo, request_slice(b, lo, hi)) for lo, hi in parts if hi > lo]
    with ThreadPoolExecutor(max_workers=len(subs)) as pool:
        t = time.perf_counter()
        list(pool.map(lambda s: oracle.run(s[1], req_index_base=s[0]), subs))
        dtm = time.perf_counter() - t
    model = cpu_model()
    desc = (f"oracle (plain C, single-threaded code) on the first {b.num_reqs} requests of the "
            f"workload ({b.num_draft_tokens} draft positions, {b.num_rows} rows): {dt:.1f} s on "
            f"1 core; {dtm:.2f} s split by requests over {len(subs)} threads on {cores} cores; "
            f"CPU {model}")
    return {"value": b.num_draft_tokens / dt, "rows_per_s": b.num_rows / dt,
            "value_multi": b.num_draft_tokens / dtm, "cores_multi": len(subs),
            "cpu_model": model, "sample": desc}


# ---------------------------------------------------------------------------------------------
def run_reference(args, world, rank):
    """The reference arm: the oracle as it stands, on this machine's host cores."""
    if rank != 0:
        return
    import oracle

    full = load_workload(args, num_reqs=2)
    t = time.perf_counter()
    oracle.run(full)
    per_req = max((time.perf_counter() - t) / 2, 1e-4)
    budget = 150.0
    n = int(max(1, min(256, budget / max(1, args.steps + args.warmup) / per_req)))
    sample = load_workload(args, num_reqs=n)
    for _ in range(args.warmup):
        oracle.run(sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run(sample)
    dt = time.perf_counter() - t0
    value = sample.num_draft_tokens * args.steps / dt
    cfg = workload_config(load_workload(args))
    cfg["reference_sample_requests_per_step"] = n
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"each step: the oracle on the first {n} requests of workload "
                                   f"{args.workload} ({sample.num_draft_tokens} draft positions)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv
    import workloads

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0:
        sv.build()
    if dist:
        dist.barrier()
    sv.lib()

    b = load_workload(args, num_reqs=args.num_reqs)
    dev = torch.device("cuda", local)
    logits_np = b.logits.view(np.int16) if b.logits.dtype == np.uint16 else b.logits
    d_logits = torch.from_numpy(logits_np).to(dev)
    dl_np = None
    if b.draft_logits is not None:
        dl_np = b.draft_logits.view(np.int16) if b.draft_logits.dtype == np.uint16 else b.draft_logits
    d_dl = torch.from_numpy(dl_np).to(dev) if dl_np is not None else None
    extras = {}
    for name in ("frequency_penalty", "output_bin_counts", "counts_row", "top_k", "top_p"):
        a = getattr(b, name, None)
        if a is not None:
            extras[name] = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d_q = torch.from_numpy(b.draft_probs).to(dev) if b.draft_probs is not None else None
    d_ids = torch.from_numpy(b.draft_ids).to(dev)
    d_cu = torch.from_numpy(b.cu_num_draft).to(dev)
    d_T = torch.from_numpy(b.temperature).to(dev)
    d_g = torch.from_numpy(b.is_greedy).to(dev)
    n, nd, kmax, V = b.num_reqs, b.num_draft_tokens, b.max_spec_len, b.vocab_size
    ctx = sv.SpecVerify(n, kmax, V, b.logits_dtype, b.draft_probs is not None, device=local,
                        draft_logits=d_dl is not None)
    if b.synthetic_rates is not None:
        ctx.set_synthetic(b.synthetic_rates)
    if args.stats_chunk:
        ctx.set_chunks(args.stats_chunk)
    outs = (torch.empty((n, kmax + 1), dtype=torch.int32, device=dev),
            torch.empty(n, dtype=torch.int32, device=dev),
            torch.empty(n, dtype=torch.int32, device=dev))
    base = rank * n  # every rank draws its own numbers

    def step():
        ctx.run(d_logits, d_ids, d_q, d_cu, d_T, d_g, b.seed, req_index_base=base,
                max_spec_len=kmax, out=outs, draft_logits=d_dl, fp64_gumbel=b.fp64_gumbel,
                **extras)

    if args.vocab_shards > 1:
        from speculative_decoding_verification_rejection_gb300.shard import ShardBackend, vocab_bounds
        sides = []
        for lo, hi in [bd for bd in vocab_bounds(V, args.vocab_shards) if bd[1] > bd[0]]:
            sl = torch.from_numpy(np.ascontiguousarray(logits_np[:, lo:hi])).to(dev)
            sq = torch.from_numpy(np.ascontiguousarray(b.draft_probs[:, lo:hi])).to(dev) \
                if b.draft_probs is not None else None
            sctx = sv.SpecVerify(n, kmax, hi - lo, b.logits_dtype, b.draft_probs is not None,
                                 device=local)
            sides.append(ShardBackend(sctx, lo, V, sl, d_ids, sq, d_cu, d_T, d_g, b.seed,
                                      req_index_base=base, max_spec_len=kmax))
        del d_logits, d_q

        def step():  # noqa: F811 - the sharded step replaces the plain one
            all_stats = torch.cat([sd.stats() for sd in sides])
            all_races = torch.cat([sd.race(all_stats, len(sides)) for sd in sides])
            out = sides[0].finish(all_races, len(sides), kmax)
            for o, t in zip(outs, out):
                o.copy_(t)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_index_for(local)) if rank == 0 else None
    if sampler:
        time.sleep(0.3)

    def load_for(seconds):
        """The same step back to back (untimed), so that the clock samples around the timed
        region see the GPU under the timed load: the timed region itself (K steps of about a
        tenth of a millisecond) is much shorter than the sampling period."""
        t = time.perf_counter()
        while time.perf_counter() - t < seconds:
            for _ in range(50):
                step()
            torch.cuda.synchronize()
        return t

    t_load0 = load_for(0.3) if sampler else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record()
    for _ in range(args.steps):
        step()
    end.record()
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    if dist:
        dist.barrier()
    elapsed_ms = start.elapsed_time(end)
    if dist:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    if sampler:
        load_for(0.3)
        t_load1 = time.perf_counter()
        time.sleep(0.1)
        sampler.stop()
    ms_per_step = elapsed_ms / args.steps
    value = world * nd / (ms_per_step / 1e3)
    mean_sampled = float(outs[1].float().mean().item())

    # per-kernel durations: CUDA events between the kernels, on the launching stream
    sharded = args.vocab_shards > 1
    kavg, calls = None, 0
    if not sharded:
        ctx.set_profiling(True)
        prof_steps = max(1, min(args.profile_steps, args.steps))
        for _ in range(prof_steps):
            step()
        torch.cuda.synchronize()
        kms, calls = ctx.get_profile()
        ctx.set_profiling(False)
        kavg = {k: v / max(calls, 1) for k, v in kms.items()}
        if args.top_k is None and args.top_p is None:
            kavg.pop("select", None)  # no selection launch: the slot holds only the events' gap

    # end to end through the host-buffer entry point: H2D of the inputs, verify, D2H of results
    e2e = None
    if sharded:
        pass  # the emulated ranks share one GPU: no end-to-end figure
    elif not args.no_e2e and (d_dl is not None or extras or b.fp64_gumbel):
        e2e = e2e_via_run(ctx, b, logits_np, dl_np, outs, base, kmax, args, world, dev, dist)
    elif not args.no_e2e:
        ctx.reserve_host_io()
        h_logits = torch.from_numpy(logits_np).pin_memory()
        h_q = torch.from_numpy(b.draft_probs).pin_memory() if b.draft_probs is not None else None
        h_ids = torch.from_numpy(b.draft_ids).pin_memory()
        h_cu = torch.from_numpy(b.cu_num_draft).pin_memory()
        h_T = torch.from_numpy(b.temperature).pin_memory()
        h_g = torch.from_numpy(b.is_greedy).pin_memory()
        h_out = (torch.empty((n, kmax + 1), dtype=torch.int32).pin_memory(),
                 torch.empty(n, dtype=torch.int32).pin_memory(),
                 torch.empty(n, dtype=torch.int32).pin_memory())

        def e2e_step():
            ctx.run_host(h_logits, h_ids, h_q, h_cu, h_T, h_g, b.seed, *h_out,
                         req_index_base=base, max_spec_len=kmax)

        for _ in range(2):
            e2e_step()
        ke = max(1, args.e2e_steps)
        if dist:
            dist.barrier()
        te = time.perf_counter()
        for _ in range(ke):
            e2e_step()
        te = time.perf_counter() - te
        if dist:
            t = torch.tensor([te], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            te = float(t.item())
        # copied every step: the logits and the small per-request arrays; the page-locked draft
        # distributions are read in place by the kernels (only the entries they need)
        h2d = h_logits.numel() * h_logits.element_size() + nd * 4 + (n + 1) * 4 + n * 4 + n
        d2h = sum(t.numel() * 4 for t in h_out)
        e2e = {"value": world * nd * ke / te, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": ke, "ms_per_step": te / ke * 1e3,
               "timing": "host wall clock around run_host (copies + kernels + stream sync)",
               "in_place": "draft_probs (page-locked host memory) read over the host link by the "
                           "verify kernel, only the entries it needs" if h_q is not None else None}
        e2e["host_link"] = host_link_ceiling(h_logits, d_logits, ke)
        e2e["link_frac"] = (h2d / (te / ke)) / 1e9 / e2e["host_link"]["h2d_gbs"]
        if not np.array_equal(h_out[0].numpy(), outs[0].cpu().numpy()):
            raise RuntimeError("host-buffer path disagrees with the device path")

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak_gbs()
    # every logit read once (R x V x element size) and one line maximum written per 64 logits;
    # in the draft-logits mode every draft logit is read once as well
    stats_bytes = b.num_rows * V * b.elem_bytes + (b.num_rows * V // 64) * b.elem_bytes
    if d_dl is not None:
        stats_bytes += nd * V * b.elem_bytes
    if b.frequency_penalty is not None:    # every request's counts row read once
        stats_bytes += n * V * 4
    if sharded:  # the whole emulated step: every shard's statistics pass reads its columns once
        achieved = stats_bytes / (ms_per_step / 1e3) / 1e9
    else:
        achieved = stats_bytes / (kavg["stats"] / 1e3) / 1e9
    plain = not extras and b.synthetic_rates is None and not sharded and not b.fp64_gumbel
    # our kernels per step: statistics + verify (+ the top-k / top-p selection, + the penalty's
    # counts-mask pass); sharded: each shard's statistics, export and race, and one finish
    launches_per_step = (3 * len(sides) + 1 if sharded else
                         sv.spec_verify_launches_per_run() + int(b.top_k is not None or b.top_p is not None)
                         + int(b.frequency_penalty is not None))
    traffic, traffic_src = (recorded_traffic("stats_kernel_workload3_draft_logits.md" if d_dl is not None
                                             else "stats_kernel_workload3.md")
                            if plain and args.workload == 3 else (None, "no ncu summary for this mode"))
    b_full, b_alg = step_bytes(b, outs[1].cpu().numpy())
    step_s = ms_per_step / 1e3
    step_roofline = {
        "bytes_full": b_full, "bytes_alg": b_alg,
        "gbs_full": b_full / step_s / 1e9, "gbs_alg": b_alg / step_s / 1e9,
        "peak_nominal_gbs": 8000.0, "frac_alg_of_nominal": b_alg / step_s / 1e9 / 8000.0,
        "frac_full_of_nominal": b_full / step_s / 1e9 / 8000.0,
        "peak_measured_gbs": peak, "frac_alg_of_measured": b_alg / step_s / 1e9 / peak,
        "note": "whole step (every kernel) against the method's bytes: logits once, plus the "
                "draft rows the method needs (alg) or every sampling request's draft rows (full)"}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        o = time_oracle(args, args.cpu_seconds)
        cpu = {"value": o["value"], "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": o["sample"], "value_multi": o["value_multi"],
               "cores_multi": o["cores_multi"], "cpu_model": o["cpu_model"]}
    clocks = None
    if sampler:
        clocks = sampler.summary(t0, t1)
        if clocks.get("note", "").startswith("timed region shorter"):
            # the window of back-to-back steps around the timed region (0.3 s on each side)
            clocks = sampler.summary(t_load0, t_load1)
            clocks["note"] = ("samples while the timed step ran back to back for 0.3 s before "
                              "and after the timed region (which is shorter than the 50 ms "
                              "sampling period), the timed region included")
    cfg = workload_config(b)
    cfg.update({"l2": "inputs larger than L2 (no flush between steps)", "parallelism":
                f"replicas x{world}" if world > 1 else "single GPU",
                "req_index_base": "rank * num_reqs"})
    if sharded:
        cfg["vocab_shards"] = f"{len(sides)} shards on 64-token boundaries, their calls in turn on one GPU"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
        "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "scope": "per kernel (the dominant one)",
                     "kernel": ("whole sharded step (every shard's kernels, the bytes of "
                                                "the statistics passes)") if sharded else
                     "sv_stats_kernel (row statistics: reads every logit once, "
                     "writes one maximum per 64-element line"
                     + ("; also reads every draft logit once)" if d_dl is not None else ")"),
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} (copy bandwidth, MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic, "traffic_source": traffic_src,
                     "algorithmic_bytes_per_launch": stats_bytes},
        "step_roofline": step_roofline,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "kernel_ms": {**kavg, "profiled_calls": calls} if kavg else None,
        "rows_per_s": world * b.num_rows / (ms_per_step / 1e3),
        # all input bytes of the batch (logits + every draft distribution) per step time; the
        # path reads every logit but only the q entries it needs
        "input_bytes_gbs": world * b.bytes_full() / (ms_per_step / 1e3) / 1e9,
        "mean_num_sampled": mean_sampled,
    }
    print(json.dumps(line), flush=True)
    ctx.close()
    if dist:
        dist.destroy_process_group()


def host_link_ceiling(h_src, d_dst, steps):
    """The plain host-to-device copy rate of the same bytes: one cudaMemcpyAsync per step of a
    page-locked host tensor into device memory (torch's non-blocking copy), timed with CUDA
    events on the current stream. What the e2e step's input copies could reach at best."""
    import torch

    for _ in range(2):
        d_dst.copy_(h_src, non_blocking=True)
    torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        d_dst.copy_(h_src, non_blocking=True)
    z.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(z) / steps
    nbytes = h_src.numel() * h_src.element_size()
    return {"h2d_gbs": nbytes / (ms / 1e3) / 1e9, "bytes": int(nbytes), "ms_per_copy": ms,
            "how": "one cudaMemcpyAsync H2D of the logits from page-locked memory per step, "
                   "CUDA events"}


def step_bytes(b, num_sampled):
    """Algorithmic bytes of one step (the method's reads): every logit row once, plus
    (full) every sampling request's draft rows once, or (alg) only the draft rows the method
    needs: the rejected row of each sampling request in draft-probability mode (its residual),
    every draft row in the draft-logits mode (q needs each row's S_d). Draft ids, outputs and
    the small per-request arrays are left out (under 0.01 %)."""
    import numpy as np

    full = b.bytes_full()
    alg = b.num_rows * b.vocab_size * b.elem_bytes
    k = np.diff(b.cu_num_draft)
    greedy = (b.is_greedy != 0) | ~(b.temperature > 0)
    if b.draft_logits is not None:
        alg = full
    elif b.draft_probs is not None and b.synthetic_rates is None:
        rejected = (~greedy) & (np.asarray(num_sampled) - 1 < k)
        alg += int(rejected.sum()) * b.vocab_size * 4
    return full, alg


def e2e_via_run(ctx, b, logits_np, dl_np, outs, base, kmax, args, world, dev, dist):
    """End to end through SpecVerify.run (draft-logits mode, logits processors): every step
    copies the step's inputs (logits, draft logits or probabilities, the per-request arrays and
    the processors' inputs) from page-locked host memory into device buffers, verifies, and
    reads the results back (host wall clock, stream synchronised)."""
    import numpy as np
    import torch

    n, nd = b.num_reqs, b.num_draft_tokens
    names = ["logits", "draft_ids", "cu_num_draft", "temperature", "is_greedy"]
    arrays = [logits_np, b.draft_ids, b.cu_num_draft, b.temperature, b.is_greedy]
    if dl_np is not None:
        names.append("draft_logits")
        arrays.append(dl_np)
    elif b.draft_probs is not None:
        names.append("draft_probs")
        arrays.append(b.draft_probs)
    for name in ("frequency_penalty", "output_bin_counts", "counts_row", "top_k", "top_p"):
        if getattr(b, name, None) is not None:
            names.append(name)
            arrays.append(getattr(b, name))
    host = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in arrays]
    devb = [torch.empty_like(h, device=dev) for h in host]
    h_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    kw = dict(zip(names, devb))

    def e2e_step():
        for h, d in zip(host, devb):
            d.copy_(h, non_blocking=True)
        ctx.run(kw["logits"], kw["draft_ids"], kw.get("draft_probs"),
                kw["cu_num_draft"], kw["temperature"], kw["is_greedy"], b.seed,
                req_index_base=base, max_spec_len=kmax, out=outs, fp64_gumbel=b.fp64_gumbel,
                **{k: v for k, v in kw.items() if k in ("draft_logits", "frequency_penalty",
                                                         "output_bin_counts", "counts_row",
                                                         "top_k", "top_p")})
        for h, o in zip(h_out, outs):
            h.copy_(o, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(2):
        e2e_step()
    ke = max(1, args.e2e_steps)
    if dist:
        dist.barrier()
    te = time.perf_counter()
    for _ in range(ke):
        e2e_step()
    te = time.perf_counter() - te
    if dist:
        t = torch.tensor([te], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        te = float(t.item())
    h2d = sum(h.numel() * h.element_size() for h in host)
    d2h = sum(h.numel() * h.element_size() for h in h_out)
    return {"value": world * nd * ke / te, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": ke, "ms_per_step": te / ke * 1e3,
            "timing": "host wall clock around H2D copies + SpecVerify.run + D2H copies + stream sync"}


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
