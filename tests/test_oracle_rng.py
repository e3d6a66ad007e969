"""Pins of the oracle's counter-based generator (Philox4x32-10 and the uniform map).

The Philox stream is checked against an independent implementation: the Philox routine of
the Triton library, run on the CPU through Triton's interpreter (seed split into
(lo32, hi32) keys, four counter words, ten rounds).
"""
import json
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
from scipy import stats

import oracle

_TRITON_SCRIPT = textwrap.dedent(r"""
    import os, sys, json
    os.environ["TRITON_INTERPRET"] = "1"
    import numpy as np, torch, triton, triton.language as tl

    @triton.jit
    def _k(c_ptr, o_ptr, seed, N: tl.constexpr):
        off = tl.arange(0, N)
        c0 = tl.load(c_ptr + off * 4 + 0).to(tl.uint32, bitcast=True)
        c1 = tl.load(c_ptr + off * 4 + 1).to(tl.uint32, bitcast=True)
        c2 = tl.load(c_ptr + off * 4 + 2).to(tl.uint32, bitcast=True)
        c3 = tl.load(c_ptr + off * 4 + 3).to(tl.uint32, bitcast=True)
        a, b, c, d = tl.random.philox(seed, c0, c1, c2, c3, 10)
        tl.store(o_ptr + off * 4 + 0, a.to(tl.int32, bitcast=True))
        tl.store(o_ptr + off * 4 + 1, b.to(tl.int32, bitcast=True))
        tl.store(o_ptr + off * 4 + 2, c.to(tl.int32, bitcast=True))
        tl.store(o_ptr + off * 4 + 3, d.to(tl.int32, bitcast=True))

    req = json.load(open(sys.argv[1]))
    res = []
    for item in req:
        ctr = np.array(item["ctr"], dtype=np.uint32).reshape(-1, 4)
        n = ctr.shape[0]
        c = torch.from_numpy(ctr.view(np.int32).copy())
        o = torch.zeros_like(c)
        _k[(1,)](c, o, item["seed"], N=n)
        res.append(o.numpy().view(np.uint32).reshape(-1).tolist())
    json.dump(res, open(sys.argv[2], "w"))
""")


def _triton_philox(requests, tmp_path):
    """requests: list of (seed, ctr[n,4]) with n a power of two. Returns list of [n,4] arrays."""
    pytest.importorskip("triton")
    pytest.importorskip("torch")
    src = tmp_path / "tphilox.py"
    src.write_text(_TRITON_SCRIPT)
    inp = tmp_path / "in.json"
    out = tmp_path / "out.json"
    inp.write_text(json.dumps([{"seed": int(s), "ctr": np.asarray(c, np.uint32).reshape(-1).tolist()}
                               for s, c in requests]))
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, str(src), str(inp), str(out)], capture_output=True,
                       text=True, env=env, timeout=600)
    if r.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + r.stderr[-400:])
    return [np.asarray(x, dtype=np.uint32).reshape(-1, 4) for x in json.loads(out.read_text())]


def test_philox_matches_triton_library(tmp_path):
    rng = np.random.default_rng(7)
    seeds = [0, 1, 0x00000000FFFFFFFF, 0x123456789ABCDEF, 0x7FFFFFFF00000001]
    reqs = []
    for s in seeds:
        ctr = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64).astype(np.uint32)
        ctr[0] = 0
        ctr[1] = 0xFFFFFFFF
        ctr[2] = [5, 0, 0, 0]       # each counter word alone
        ctr[3] = [0, 5, 0, 0]
        ctr[4] = [0, 0, 5, 0]
        ctr[5] = [0, 0, 0, 5]
        reqs.append((s, ctr))
    ref = _triton_philox(reqs, tmp_path)
    for (s, ctr), want in zip(reqs, ref):
        key = [s & 0xFFFFFFFF, s >> 32]
        got = np.stack([oracle.philox(c, key) for c in ctr])
        np.testing.assert_array_equal(got, want, err_msg=f"seed {s:#x}")


def _u(w):
    return ((np.asarray(w, np.uint64) >> 9).astype(np.float64) + 0.5) * 2.0**-23


def test_race_clock_layout_matches_triton(tmp_path):
    """The race clock of token v (group g = v >> 6, slot s = v & 63) at (request i, position j):
    counter (g, j, i, 8) gives W (word 0) and the argmin slot a (word 1 & 63); E_min = -ln(W)/64;
    slot s != a adds -ln U_s, U_s word s & 3 of counter (g, j, i, 9 + s // 4)."""
    seed, j, i = 0xDEADBEEF12345, 3, 17
    groups = [(0, 1, 2), (3, 4, 5)]                # 17 calls per group; 64 counters per request
    reqs = []
    for gs in groups:
        ctr = np.array([[g, j, i, 8 + k] for g in gs for k in range(17)], dtype=np.uint32)
        reqs.append((seed, np.vstack([ctr, np.zeros((64 - ctr.shape[0], 4), np.uint32)])))
    words = _triton_philox(reqs, tmp_path)
    nblk = sum(len(gs) for gs in groups)
    want = np.empty(64 * nblk)
    for gs, w in zip(groups, words):
        for k, g in enumerate(gs):
            head = w[17 * k]
            emin = -np.log(_u(head[0])) / 64.0
            a = int(head[1]) & 63
            for s_ in range(64):
                v = 64 * g + s_
                want[v] = emin if s_ == a else emin - np.log(_u(w[17 * k + 1 + s_ // 4][s_ % 4]))
    got = oracle.race_clocks(seed, j, i, 64 * nblk).astype(np.float64)
    np.testing.assert_allclose(got, want, rtol=2e-6)


def test_uniform_map_extremes_and_exactness():
    assert oracle.uniform_from_word(0) == 2.0**-24
    assert oracle.uniform_from_word(0xFFFFFFFF) == 1.0 - 2.0**-24
    assert oracle.uniform_from_word(0x1FF) == 2.0**-24          # low 9 bits are dropped
    assert oracle.uniform_from_word(0x200) == 3 * 2.0**-24
    w = np.random.default_rng(3).integers(0, 2**32, 2000, dtype=np.uint64)
    for x in w[:200]:
        u = oracle.uniform_from_word(int(x))
        assert 0.0 < u < 1.0
        assert u == ((int(x) >> 9) + 0.5) / 2**23                # exact in binary32


def test_uniforms_are_uniform_and_uncorrelated():
    u = np.array([oracle.uniform(99, c, 0, 0, 0, w) for c in range(25_000) for w in range(4)])
    counts, _ = np.histogram(u, bins=100, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-3
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    assert abs(np.corrcoef(u[:-1], u[1:])[0, 1]) < 0.02        # words of one call and neighbours
    v = np.array([oracle.uniform(99, c, 0, 1, 0, 0) for c in range(25_000)])  # another request
    assert abs(np.corrcoef(u[::4], v)[0, 1]) < 0.03


def test_race_clocks_are_iid_exponential():
    """The group construction (minimum of 64 and memoryless excesses) must give i.i.d. Exp(1)
    clocks: the marginal of every slot, the argmin slot uniform, no correlation in a group."""
    n = 64 * 10_000
    e = oracle.race_clocks(2024, 1, 5, n).astype(np.float64)
    assert stats.kstest(e, "expon").pvalue > 1e-3
    blocks = e.reshape(-1, 64)
    for s_ in (0, 5, 63):
        assert stats.kstest(blocks[:, s_], "expon").pvalue > 1e-3
    argmin = np.bincount(blocks.argmin(axis=1), minlength=64)
    assert stats.chisquare(argmin).pvalue > 1e-3
    assert stats.kstest(blocks.min(axis=1) * 64, "expon").pvalue > 1e-3   # min of 64 ~ Exp(64)
    c = np.corrcoef(blocks[:, 2], blocks[:, 41])[0, 1]
    assert abs(c) < 0.02
    other = oracle.race_clocks(2024, 2, 5, 64 * 1250).astype(np.float64)  # another position
    assert abs(np.corrcoef(e[: other.size], other)[0, 1]) < 0.03
