"""GPU-vs-oracle comparison used by the -m gpu tests and the smoke check.

Token ids and accept lengths must match bit for bit. The only exception is a request whose
outputs differ after a decision the oracle calls too close to call: an acceptance test with
|u - p/q| < 1e-6 at a position both sides evaluated, or a residual race whose two best keys
are closer than 1e-6 (the residual depends on the row's sum of exponentials S, which the two
sides accumulate in different orders), or a top-p boundary within 1e-6 of the total mass at a
row both sides used (the kept mass is summed in binary32 on the GPU). Such a request is a
counted tie and the rest of it is not compared. The row statistics must match: m and the
argmax exactly, S (the kept mass under top-k / top-p) to 1e-5 relative, except at rows whose
top-p boundary is that close, where S is not compared (the boundary group may fall either way).
"""
from __future__ import annotations

import numpy as np

TIE_MARGIN = 1e-6
SEL_MARGIN = 1e-6
S_RTOL = 1e-5
RACE_NONE = 0


def to_device(batch, device="cuda:0"):
    import torch

    logits = np.ascontiguousarray(batch.logits)
    lt = torch.from_numpy(logits.view(np.int16) if logits.dtype == np.uint16 else logits).to(device)
    q = None
    if batch.draft_probs is not None:
        q = torch.from_numpy(np.ascontiguousarray(batch.draft_probs, np.float32)).to(device)
    dl = None
    if getattr(batch, "draft_logits", None) is not None:
        d = np.ascontiguousarray(batch.draft_logits)
        dl = torch.from_numpy(d.view(np.int16) if d.dtype == np.uint16 else d).to(device)
    pp = None
    if getattr(batch, "partial_prefill", None) is not None:
        pp = torch.from_numpy(np.ascontiguousarray(batch.partial_prefill, np.uint8)).to(device)
    extra = {}
    for name, dt in (("frequency_penalty", np.float32), ("output_bin_counts", np.int32),
                     ("counts_row", np.int32), ("top_k", np.int32), ("top_p", np.float32)):
        a = getattr(batch, name, None)
        extra[name] = None if a is None else torch.from_numpy(np.ascontiguousarray(a, dt)).to(device)
    return dict(
        **extra,
        logits=lt,
        draft_logits=dl,
        partial_prefill=pp,
        draft_ids=torch.from_numpy(np.ascontiguousarray(batch.draft_ids, np.int32)).to(device),
        draft_probs=q,
        cu_num_draft=torch.from_numpy(np.ascontiguousarray(batch.cu_num_draft, np.int32)).to(device),
        temperature=torch.from_numpy(np.ascontiguousarray(batch.temperature, np.float32)).to(device),
        is_greedy=torch.from_numpy(np.ascontiguousarray(batch.is_greedy, np.uint8)).to(device),
    )


CANARY_PAD = 64            # 4-byte words of sentinel before and after every output buffer
CANARY_WORD = -0x21524111  # 0xDEADBEEF


def canary_buffer(shape, dtype, device):
    """An output tensor of `shape` inside a larger buffer whose CANARY_PAD words before and
    after it hold CANARY_WORD: (buffer, view). A kernel writing past either end of the output
    changes a canary (compute-sanitizer is not available on the GPU machines; this catches
    out-of-bounds stores into the neighbours of every output)."""
    import torch

    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + 2 * CANARY_PAD,), CANARY_WORD, dtype=torch.int32, device=device)
    view = buf[CANARY_PAD:CANARY_PAD + n]
    if dtype != torch.int32:
        view = view.view(dtype)
    return buf, view.view(shape)


def check_canaries(buf, name):
    import torch

    pad = torch.cat([buf[:CANARY_PAD], buf[-CANARY_PAD:]]).cpu().numpy()
    bad = np.flatnonzero(pad != CANARY_WORD)
    assert bad.size == 0, f"{name}: {bad.size} canary words overwritten (first at {bad[:4]})"


def gpu_run(batch, ctx=None, *, max_spec_len=None, req_index_base=0, seed=None, chunks=None,
            device="cuda:0"):
    """Run the library on a workloads.Batch (through the draft-logits entry point when the batch
    carries draft logits); returns numpy outputs incl. row stats."""
    import torch

    import speculative_decoding_verification_rejection_gb300 as sv

    kmax = batch.max_spec_len if max_spec_len is None else max_spec_len
    own = ctx is None
    has_dl = getattr(batch, "draft_logits", None) is not None
    if own:
        ctx = sv.SpecVerify(max(batch.num_reqs, 1), max(kmax, 0), batch.vocab_size,
                            batch.logits_dtype, batch.draft_probs is not None,
                            device=torch.device(device).index or 0, draft_logits=has_dl)
    if chunks:
        ctx.set_chunks(chunks)
    rates = getattr(batch, "synthetic_rates", None)
    ctx.set_synthetic([] if rates is None else rates)
    d = to_device(batch, device)
    n, R = batch.num_reqs, batch.num_rows
    shapes = (((n, kmax + 1), torch.int32), ((n,), torch.int32), ((n,), torch.int32),
              ((R,), torch.float32), ((R,), torch.float32), ((R,), torch.int32))
    padded = [canary_buffer(shape, dt, device) for shape, dt in shapes]
    views = [v for _, v in padded]
    outs = ctx.run(d["logits"], d["draft_ids"], d["draft_probs"], d["cu_num_draft"],
                   d["temperature"], d["is_greedy"], batch.seed if seed is None else seed,
                   req_index_base=req_index_base, max_spec_len=kmax, row_stats=True,
                   out=tuple(views[:3]), stats_out=tuple(views[3:]),
                   draft_logits=d["draft_logits"], partial_prefill=d["partial_prefill"],
                   frequency_penalty=d["frequency_penalty"], output_bin_counts=d["output_bin_counts"],
                   counts_row=d["counts_row"], top_k=d["top_k"], top_p=d["top_p"],
                   fp64_gumbel=bool(getattr(batch, "fp64_gumbel", False)))
    torch.cuda.synchronize()
    names = ("sampled", "num_sampled", "num_rejected", "row_max", "row_sumexp", "row_argmax")
    for name, (buf, _) in zip(names, padded):
        check_canaries(buf, name)
    res = {k: v.cpu().numpy() for k, v in zip(names, outs)}
    res["error_word"] = ctx.last_error()
    if own:
        ctx.close()
    return res


def compare(batch, gpu: dict, ref: dict) -> dict:
    """Compare GPU outputs with the oracle's. Returns counts; raises AssertionError with the
    first real mismatches."""
    cu = batch.cu_num_draft
    n = batch.num_reqs
    ties, bad = [], []
    for i in range(n):
        if (gpu["num_sampled"][i] == ref["num_sampled"][i]
                and gpu["num_rejected"][i] == ref["num_rejected"][i]
                and np.array_equal(gpu["sampled"][i], ref["sampled"][i])):
            continue
        js_ref = int(ref["jstar"][i])
        js_gpu = int(gpu["num_sampled"][i]) - 1
        upto = min(js_ref, js_gpu)
        m = ref["accept_margin"][cu[i]:cu[i] + max(upto, -1) + 1]
        m = m[~np.isnan(m)]
        closest = float(m.min()) if m.size else np.inf
        if js_ref == js_gpu and ref["race_kind"][i] != RACE_NONE:
            closest = min(closest, float(ref["race_gap"][i]))
        sel = ref.get("row_select_margin")
        if sel is not None and upto >= 0:
            r0 = cu[i] + i
            if np.min(sel[r0:r0 + upto + 1]) < SEL_MARGIN:
                closest = min(closest, 0.0)
        (ties if closest < TIE_MARGIN else bad).append((i, closest))
    R = batch.num_rows
    stats_ok = dict(
        row_max=bool(np.array_equal(gpu["row_max"][:R], ref["row_max"][:R])),
        row_argmax=bool(np.array_equal(gpu["row_argmax"][:R], ref["row_argmax"][:R])),
    )
    rel = np.abs(gpu["row_sumexp"][:R].astype(np.float64) - ref["row_sumexp"][:R]) / \
        np.maximum(np.abs(ref["row_sumexp"][:R].astype(np.float64)), 1e-30)
    sel = ref.get("row_select_margin")
    if sel is not None:                       # a top-p boundary too close to call: S is loose
        rel = np.where(sel[:R] < SEL_MARGIN, 0.0, rel)
    stats_ok["row_sumexp"] = bool(np.all(rel <= S_RTOL))
    out = dict(requests=n, positions=int(cu[-1]), ties=len(ties), mismatches=bad,
               max_sumexp_rel=float(rel.max()) if R else 0.0, **stats_ok)
    return out


def assert_parity(batch, gpu: dict, ref: dict) -> dict:
    r = compare(batch, gpu, ref)
    assert not r["mismatches"], f"{len(r['mismatches'])} requests differ: {r['mismatches'][:5]}"
    assert r["row_max"], "row max differs"
    assert r["row_argmax"], "row argmax differs"
    assert r["row_sumexp"], f"row sum of exponentials off by {r['max_sumexp_rel']:.3g} relative"
    assert r["ties"] <= 1e-5 * max(r["positions"], 1), f"{r['ties']} counted ties"
    return r
