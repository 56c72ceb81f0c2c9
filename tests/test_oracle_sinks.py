"""Pins of the oracle's attention sinks (CPU only).

The pages name attention sinks only where "RBLN Attention modes" (Full
Attention, kernel choice) picks flash attention for a layer that has them;
they give no formula.  The reading: one logit per query head joins the
softmax normaliser as a term with no value,
    out = sum_k e^{s_k} V_k / (e^{sink_h} + sum_k e^{s_k}),
in the units of s_k = scale * q.k.  Pinned, independently of the oracle's own
code, by:
  - a sink of -inf is exactly no sink;
  - the dense brute force (tests/brute.py), which appends the sink as one more
    key whose score is the sink and whose value row is zero;
  - a closed form: with scale 0 every visible score is 0, so
    out = sum of the n visible V rows / (n + e^{sink});
  - split == unsplit with sinks (the sink enters the partition merge);
  - a sink far above every score: out is 0 and lse is the sink.
Planted mistakes in the oracle's sink code must each fail one of them."""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads as W
from brute import brute_attention
from cases import case_args, host_arrays, small_spec

HERE = os.path.dirname(os.path.abspath(__file__))


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    ok = ~np.isnan(b)
    if np.isnan(a[ok]).any():
        return math.inf
    return float(np.max(np.abs(a[ok] - b[ok])) / max(1.0, np.max(np.abs(b[ok]))))


def _oracle(case, sinks, lib=None, **over):
    q, kv, bt, sl, qsl = host_arrays(case)
    kw = case_args(case)
    kw.update(over)
    return oracle.ref_varlen(q, kv, bt, sl, qsl, sinks=sinks, lib=lib, **kw)


def _sinks(H, seed):
    rng = np.random.default_rng(seed)
    s = rng.normal(0.0, 2.0, H).astype(np.float32)
    s[0] = 6.0  # above most scores: its weight dominates some rows
    return s


def sink_failures(lib):
    bad = []
    specs = [small_spec(301, H=4, Hkv=2, d=16, n_req=4, max_s=80),
             small_spec(302, H=8, Hkv=2, d=16, n_req=4, window=9, max_s=80),
             small_spec(303, H=4, Hkv=2, d=16, n_req=3, kv_dtype=1, max_s=80)]
    for sp in specs:
        case = W.make_case(sp)
        H = sp.num_heads
        try:
            base = _oracle(case, None, lib=lib)
            none = _oracle(case, np.full(H, -np.inf, np.float32), lib=lib)
            sinks = _sinks(H, sp.seed)
            out, lse = _oracle(case, sinks, lib=lib)
            out3, lse3 = _oracle(case, sinks, lib=lib, num_splits=3)
        except oracle.OracleError:
            bad.append(sp.name + ":error")
            continue
        if not (np.array_equal(base[0], none[0], equal_nan=True) and
                np.array_equal(base[1], none[1], equal_nan=True)):
            bad.append(sp.name + ":minus-inf")
        ob, lb = brute_attention(case.q, case.kv_cache, case.block_table, case.seq_lens,
                                 case.query_start_loc, sinks=sinks, **case_args(case))
        if _rel(out, ob) > 1e-12 or _rel(lse, lb) > 1e-12:
            bad.append(sp.name + ":brute")
        if _rel(out3, out) > 1e-12 or _rel(lse3, lse) > 1e-12:
            bad.append(sp.name + ":split")
    # closed form at scale 0: out = sum V / (n + e^sink)
    sp = small_spec(304, H=2, Hkv=1, d=8, n_req=2, max_s=40, kinds=("decode",), scale=0.0)
    case = W.make_case(sp)
    sinks = np.array([0.5, -1.25], np.float32)
    try:
        out, lse = _oracle(case, sinks, lib=lib)
    except oracle.OracleError:
        return bad + ["closed-form:error"]
    kv = case.kv_cache.cpu().float().double().numpy()
    bt = case.block_table.cpu().numpy()
    qsl = case.query_start_loc.cpu().numpy()
    for r, s in enumerate(sp.seq_lens):
        t = int(qsl[r])
        V = np.stack([kv[1, bt[r, k // 16], k % 16, 0] for k in range(s)])
        for h in range(2):
            den = s + math.exp(float(sinks[h]))
            if (np.max(np.abs(out[t, h] - V.sum(0) / den)) > 1e-12 or
                    abs(lse[t, h] - math.log(den)) > 1e-12):
                bad.append("closed-form")
    # a sink far above every score
    sp = small_spec(305, H=2, Hkv=1, d=8, n_req=2, max_s=40)
    case = W.make_case(sp)
    try:
        out, lse = _oracle(case, np.array([1e4, 1e4], np.float32), lib=lib)
        out3, lse3 = _oracle(case, np.array([1e4, 1e4], np.float32), lib=lib, num_splits=2)
    except oracle.OracleError:
        return bad + ["large:error"]
    rows = ~np.isnan(lse)
    for o, l in ((out, lse), (out3, lse3)):
        if np.any(o[rows] != 0.0) or np.any(l[rows] != 1e4):
            bad.append("large-sink")
    return bad


def test_sink_pins_pass_on_the_oracle():
    assert sink_failures(None) == []


MUTATIONS = {
    "sink_scaled": ("const double sink = jb->sinks ? (double)jb->sinks[h] : -INFINITY;",
                    "const double sink = jb->sinks ? (double)jb->sinks[h] * jb->scale : -INFINITY;"),
    "sink_head_fixed": ("const double sink = jb->sinks ? (double)jb->sinks[h] : -INFINITY;",
                        "const double sink = jb->sinks ? (double)jb->sinks[0] : -INFINITY;"),
    "sink_left_out_of_denominator": ("double denom = has_sink ? exp(sink - m) : 0.0;",
                                     "double denom = 0.0;"),
    "sink_not_in_max": ("if (has_sink && (!any || sink > m)) m = sink;",
                        "if (has_sink && !any) m = sink;"),
    "sink_left_out_of_merge": ("if (sink > -INFINITY) sum += exp(sink - lse_max);", ""),
    "sink_counted_per_partition": (
        "attend_range(jb, r, qv, g, p, kb, ke, -INFINITY, scores,",
        "attend_range(jb, r, qv, g, p, kb, ke, sink, scores,"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_sink_mistakes_are_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "pattn_ref.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
    (tmp_path / "mut.c").write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(tmp_path / "mut.c"), "-lm"], check=True)
    lib = oracle.bind(str(so))
    assert sink_failures(lib), f"{name} went unnoticed"
