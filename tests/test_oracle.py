"""Pins for the float64 oracle (CPU only).

The oracle is checked against things other than itself: hand-derived closed
forms (tests/golden/closed_forms.json), a dense brute force with a different
structure (tests/brute.py), PyTorch's scaled_dot_product_attention in float64,
torch's own bf16 / e4m3 decoders, and invariants that hold for exact attention
(block shuffles, window >= seq_len, split == unsplit, MHA reduction, prefix
consistency).  ``test_planted_mistakes`` plants plausible mistakes in a copy
of the oracle source and checks that these pins catch each one.
"""
import json
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from brute import brute_attention
from cases import case_args, host_arrays, shuffle_blocks, small_spec

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "closed_forms.json")


def run_oracle(case, lib=None, **over):
    q, kv, bt, sl, qsl = host_arrays(case)
    kw = case_args(case)
    kw.update(over)
    return oracle.ref_varlen(q, kv, bt, sl, qsl, lib=lib, **kw)


def run_brute(case):
    return brute_attention(case.q, case.kv_cache, case.block_table, case.seq_lens,
                           case.query_start_loc, **case_args(case))


def rel_err(a, b):
    a, b = np.asarray(a), np.asarray(b)
    ok = ~np.isnan(b)
    if np.isnan(a).sum() != (~ok).sum() or np.isnan(a[ok]).any():
        return math.inf
    if not ok.any():
        return 0.0
    return float(np.max(np.abs(a[ok] - b[ok])) / max(1.0, np.max(np.abs(b[ok]))))


# ----------------------------------------------------------------- goldens

def _eval_num(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, {"e": math.e, "log": math.log}))
    return float(x)


def golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)


def golden_to_case(g):
    """Page a fixture's dense per-request K/V into a cache through its block ids."""
    H, Hkv, d, bs = g["H"], g["Hkv"], g["d"], g["bs"]
    kv_dtype = g.get("kv_dtype", 0)
    pool = g["pool"]
    if kv_dtype == 0:
        kv = torch.zeros((2, pool, bs, Hkv, d), dtype=torch.bfloat16)
    else:
        kv = torch.zeros((2, pool, bs, Hkv, d), dtype=torch.uint8)
    mb = max(len(b) for b in g["blocks"])
    bt = torch.zeros((len(g["q_lens"]), mb), dtype=torch.int32)
    for r, blocks in enumerate(g["blocks"]):
        bt[r, :len(blocks)] = torch.tensor(blocks, dtype=torch.int32)
        for kv_i, key in ((0, "k"), (1, "v")):
            if kv_dtype == 0:
                dense = torch.tensor(g[key][r], dtype=torch.float32).to(torch.bfloat16)
            else:
                dense = torch.tensor(g[key + "_bytes"][r], dtype=torch.uint8)
            for kk in range(dense.shape[0]):
                kv[kv_i, blocks[kk // bs], kk % bs] = dense[kk]
    q = torch.tensor(g["q"], dtype=torch.float32).to(torch.bfloat16)
    qsl = torch.zeros(len(g["q_lens"]) + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(torch.tensor(g["q_lens"]), 0)
    spec = W.CaseSpec(g["name"], g["q_lens"], g["seq_lens"], H, Hkv, d, bs,
                      window=g["window"], causal=g["causal"], kv_dtype=kv_dtype,
                      scale=g["scale"])
    return W.Case(spec=spec, q=q, kv_cache=kv, block_table=bt,
                  seq_lens=torch.tensor(g["seq_lens"], dtype=torch.int32),
                  query_start_loc=qsl, scale=float(np.float32(g["scale"])),
                  kv_scale=tuple(g.get("kv_scale", (1.0, 1.0))))


def golden_failures(lib=None):
    bad = []
    for g in golden_cases():
        case = golden_to_case(g)
        out, lse = run_oracle(case, lib=lib)
        exp_out = np.vectorize(_eval_num)(np.array(g["out"], dtype=object)).astype(float)
        if not np.allclose(out, exp_out, rtol=1e-12, atol=1e-12):
            bad.append(g["name"] + ":out")
        if g["lse"] is not None:
            exp_lse = np.vectorize(_eval_num)(np.array(g["lse"], dtype=object)).astype(float)
            if not np.allclose(lse, exp_lse, rtol=1e-12, atol=1e-12):
                bad.append(g["name"] + ":lse")
    return bad


@pytest.mark.parametrize("name", [g["name"] for g in golden_cases()])
def test_golden_closed_forms(name):
    g = [x for x in golden_cases() if x["name"] == name][0]
    case = golden_to_case(g)
    out, lse = run_oracle(case)
    exp_out = np.vectorize(_eval_num)(np.array(g["out"], dtype=object)).astype(float)
    np.testing.assert_allclose(out, exp_out, rtol=1e-12, atol=1e-12)
    if g["lse"] is not None:
        exp_lse = np.vectorize(_eval_num)(np.array(g["lse"], dtype=object)).astype(float)
        np.testing.assert_allclose(lse, exp_lse, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- decoders

def test_bf16_decoder_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))


def test_e4m3_decoder_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6
    assert got[0x38] == 1.0 and got[0xB8] == -1.0


# ----------------------------------------------------------------- brute force

BRUTE_PARAMS = []
for i in range(36):
    H, Hkv = [(4, 2), (4, 4), (8, 2), (4, 1)][i % 4]
    d = [8, 16, 64][i % 3]
    bs = [16, 32][(i // 3) % 2]
    window = [0, 0, 1, 3, 16, 1000][i % 6]
    causal = 0 if (i % 9 == 4 and window == 0) else 1
    kv_dtype = 1 if i % 5 == 2 else 0
    BRUTE_PARAMS.append((i, H, Hkv, d, bs, window, causal, kv_dtype))


@pytest.mark.parametrize("i,H,Hkv,d,bs,window,causal,kv_dtype", BRUTE_PARAMS)
def test_oracle_matches_brute_force(i, H, Hkv, d, bs, window, causal, kv_dtype):
    spec = small_spec(100 + i, H=H, Hkv=Hkv, d=d, bs=bs, window=window, causal=causal,
                      kv_dtype=kv_dtype, n_req=4,
                      kinds=("prefill", "decode", "chunk", "empty"))
    case = W.make_case(spec)
    out, lse = run_oracle(case)
    ob, lb = run_brute(case)
    assert rel_err(out, ob) <= 1e-12
    assert rel_err(lse, lb) <= 1e-12


def _sdpa(case):
    """torch SDPA (float64, CPU) per request, GQA heads expanded, an explicit
    boolean mask for the bottom-right causal / window rule."""
    s = case.spec
    q = case.q.to(torch.float64)
    G = s.num_heads // s.num_kv_heads
    outs = torch.full(q.shape, float("nan"), dtype=torch.float64)
    kvd = case.kv_cache.to(torch.float64)
    for r in range(case.num_seqs):
        t0, t1 = int(case.query_start_loc[r]), int(case.query_start_loc[r + 1])
        sl = int(case.seq_lens[r])
        if t1 == t0:
            continue
        nb = (sl + s.block_size - 1) // s.block_size
        blk = case.block_table[r, :nb].long()
        K = kvd[0, blk].reshape(-1, s.num_kv_heads, s.head_size)[:sl]
        V = kvd[1, blk].reshape(-1, s.num_kv_heads, s.head_size)[:sl]
        K = K.repeat_interleave(G, dim=1).transpose(0, 1)
        V = V.repeat_interleave(G, dim=1).transpose(0, 1)
        Q = q[t0:t1].transpose(0, 1)
        pos = torch.arange(sl - (t1 - t0), sl)[:, None]
        key = torch.arange(sl)[None, :]
        mask = torch.ones(t1 - t0, sl, dtype=torch.bool)
        if s.causal:
            mask &= key <= pos
        if s.window > 0:
            mask &= (pos - key) < s.window
        o = torch.nn.functional.scaled_dot_product_attention(
            Q, K, V, attn_mask=mask, scale=case.scale)
        outs[t0:t1] = o.transpose(0, 1)
    return outs.numpy()


@pytest.mark.parametrize("seed,window", [(7, 0), (8, 0), (9, 5), (10, 33)])
def test_oracle_matches_torch_sdpa(seed, window):
    spec = small_spec(seed, H=8, Hkv=2, d=64, bs=16, window=window, n_req=4, max_s=90)
    case = W.make_case(spec)
    out, _ = run_oracle(case)
    assert rel_err(out, _sdpa(case)) <= 1e-12


def test_oracle_matches_torch_sdpa_noncausal():
    spec = small_spec(11, H=4, Hkv=4, d=32, bs=16, causal=0, n_req=3, max_s=50)
    case = W.make_case(spec)
    out, _ = run_oracle(case)
    assert rel_err(out, _sdpa(case)) <= 1e-12


# ----------------------------------------------------------------- special cases

def test_tiny_mixed_first_row_is_v0():
    """Workload 1: request 0, row 0 sits at position 0 and sees only key 0."""
    case = W.make_case(W.config_spec(1))
    out, lse = run_oracle(case)
    blk = int(case.block_table[0, 0])
    for h in range(4):
        v0 = case.kv_cache[1, blk, 0, h // 2].to(torch.float64).numpy()
        assert np.array_equal(out[0, h], v0)


def test_constant_v_rows():
    spec = small_spec(21, H=4, Hkv=2, d=16, n_req=4, window=5)
    case = W.make_case(spec)
    v = torch.tensor([0.5 * (j - 7) for j in range(16)], dtype=torch.bfloat16)
    case.kv_cache[1] = v
    out, _ = run_oracle(case)
    rows = ~np.isnan(out[:, 0, 0])
    assert np.allclose(out[rows], v.to(torch.float64).numpy(), rtol=0, atol=1e-13)


def test_zero_query_gives_mean_of_visible_v():
    spec = small_spec(22, H=2, Hkv=1, d=8, n_req=3, window=4)
    case = W.make_case(spec)
    case.q.zero_()
    out, _ = run_oracle(case)
    ob, _ = run_brute(case)
    # brute force with scale = 0 is a plain mean; compare the two definitions
    case0 = W.Case(spec=spec, q=case.q, kv_cache=case.kv_cache,
                   block_table=case.block_table, seq_lens=case.seq_lens,
                   query_start_loc=case.query_start_loc, scale=0.0)
    out0, _ = run_oracle(case0)
    assert rel_err(out, out0) <= 1e-13 and rel_err(out, ob) <= 1e-12
    # and directly: mean over the window of the decode / last row
    bs = spec.block_size
    for r in range(case.num_seqs):
        t1 = int(case.query_start_loc[r + 1])
        if t1 == int(case.query_start_loc[r]):
            continue
        s = int(case.seq_lens[r])
        keys = range(max(0, s - 4), s)
        vs = [case.kv_cache[1, int(case.block_table[r, k // bs]), k % bs, 0]
              .to(torch.float64).numpy() for k in keys]
        assert np.allclose(out[t1 - 1, 0], np.mean(vs, axis=0), atol=1e-13)


# ----------------------------------------------------------------- invariants

@pytest.mark.parametrize("seed", [31, 32, 33])
def test_block_shuffle_is_bitwise_invariant(seed):
    case = W.make_case(small_spec(seed, n_req=4, extra_pool=6, max_s=100))
    a, la = run_oracle(case)
    b, lb = run_oracle(shuffle_blocks(case, seed + 1))
    assert np.array_equal(a, b, equal_nan=True) and np.array_equal(la, lb, equal_nan=True)


def test_window_at_least_seq_len_equals_full():
    spec = small_spec(41, n_req=4, max_s=60)
    case = W.make_case(spec)
    full, lf = run_oracle(case)
    for w in (60, 61, 1000):
        win, lw = run_oracle(case, window=w)
        assert np.array_equal(full, win, equal_nan=True)
        assert np.array_equal(lf, lw, equal_nan=True)


@pytest.mark.parametrize("splits", [2, 3, 5, 16])
def test_split_merge_equals_unsplit(splits):
    spec = small_spec(51, n_req=5, max_s=200, window=70, kinds=("decode", "chunk"))
    case = W.make_case(spec)
    a, la = run_oracle(case)
    b, lb = run_oracle(case, num_splits=splits)
    assert rel_err(b, a) <= 1e-12 and rel_err(lb, la) <= 1e-12


def test_mha_reduction_of_gqa():
    """GQA with Hkv = 2 equals MHA whose KV heads are copies (0, 0, 1, 1)."""
    spec = small_spec(61, H=4, Hkv=2, d=16, n_req=3)
    case = W.make_case(spec)
    mspec = W.CaseSpec(**{**spec.__dict__, "num_kv_heads": 4})
    mcase = W.Case(spec=mspec, q=case.q,
                   kv_cache=case.kv_cache.repeat_interleave(2, dim=3).contiguous(),
                   block_table=case.block_table, seq_lens=case.seq_lens,
                   query_start_loc=case.query_start_loc, scale=case.scale)
    a, _ = run_oracle(case)
    b, _ = run_oracle(mcase)
    assert np.array_equal(a, b, equal_nan=True)


def test_prefix_consistency_decode_and_chunk():
    """A decode at seq_len s equals row s-1 of a full prefill over the same
    cache; a chunk of c rows on s - c cached tokens equals the last c rows."""
    s_len, c = 45, 13
    spec = W.CaseSpec("pf", [s_len], [s_len], 4, 2, 16, 16, seed=71)
    full = W.make_case(spec)
    a, _ = run_oracle(full)
    for ql in (1, c):
        sub = W.Case(spec=W.CaseSpec("pc", [ql], [s_len], 4, 2, 16, 16, seed=71),
                     q=full.q[s_len - ql:].clone(), kv_cache=full.kv_cache,
                     block_table=full.block_table, seq_lens=full.seq_lens,
                     query_start_loc=torch.tensor([0, ql], dtype=torch.int32),
                     scale=full.scale)
        b, _ = run_oracle(sub)
        assert np.array_equal(b, a[s_len - ql:])


def test_poisoned_unused_slots_do_not_matter():
    spec = small_spec(81, n_req=4, extra_pool=3, max_s=70)
    case = W.make_case(spec)
    a, _ = run_oracle(case)
    kv = case.kv_cache.clone()
    used = set()
    for r in range(case.num_seqs):
        s = int(case.seq_lens[r])
        nb = (s + 15) // 16
        for j in range(nb):
            used.add(int(case.block_table[r, j]))
        last = int(case.block_table[r, nb - 1])
        kv[:, last, s - (nb - 1) * 16:] = float("nan")
    for b in range(kv.shape[1]):
        if b not in used:
            kv[:, b] = float("nan")
    pc = W.Case(spec=spec, q=case.q, kv_cache=kv, block_table=case.block_table,
                seq_lens=case.seq_lens, query_start_loc=case.query_start_loc,
                scale=case.scale)
    b, _ = run_oracle(pc)
    assert np.array_equal(a, b, equal_nan=True)


def test_metadata_errors_are_reported():
    case = W.make_case(small_spec(91, n_req=2))
    q, kv, bt, sl, qsl = host_arrays(case)
    bad_sl = sl.copy()
    bad_sl[0] = 0 if (qsl[1] - qsl[0]) > 0 else bad_sl[0]
    if (qsl[1] - qsl[0]) > 0:
        with pytest.raises(oracle.OracleError):
            oracle.ref_varlen(q, kv, bt, bad_sl, qsl, **case_args(case))
    bad_bt = bt.copy()
    bad_bt[0, 0] = kv.shape[1]
    with pytest.raises(oracle.OracleError):
        oracle.ref_varlen(q, kv, bad_bt, sl, qsl, **case_args(case))


# ----------------------------------------------------------------- planted mistakes

MUTATIONS = {
    "causal_off_by_one": ("if (jb->causal && k > p)", "if (jb->causal && k >= p)"),
    "window_off_by_one": ("p - k >= jb->window", "p - k > jb->window"),
    "gqa_interleaved": ("int g = h / (jb->num_heads / jb->num_kv_heads);",
                        "int g = h % jb->num_kv_heads;"),
    "scale_dropped": ("scores[k] = jb->scale * dot;", "scores[k] = dot;"),
    "exp_sign": ("double w = exp(scores[k] - m);", "double w = exp(m - scores[k]);"),
    "context_offset_dropped": ("p = ctx + i;", "p = i;"),
    "v_read_from_k": ("o[j] += w * cache_elem(jb, 1,", "o[j] += w * cache_elem(jb, 0,"),
    "kv_scales_swapped": ("(kv_index == 0 ? jb->k_scale : jb->v_scale)",
                          "(kv_index == 0 ? jb->v_scale : jb->k_scale)"),
    "e4m3_bias": ("mag = ldexp(1.0 + (double)m / 8.0, e - 7);",
                  "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_subnormal": ("mag = ldexp((double)m, -9);", "mag = ldexp((double)m, -10);"),
    "lse_missing_max": ("return m + log(denom);", "return log(denom);"),
    "merge_weight": ("double wgt = exp(lse_p[sp] - lse);",
                     "double wgt = exp(lse_p[sp] - lse_max);"),
    "head_stride": ("jb->q[((int64_t)t * jb->num_heads + h) * d + j]",
                    "jb->q[((int64_t)t * jb->num_heads + (h % 2)) * d + j]"),
    "slot_index": ("int blk = bt[k / bs], slot = k % bs;\n    double w",
                   "int blk = bt[k / bs], slot = (k + 1) % bs;\n    double w"),
}


def pin_failures(lib):
    """Run a compact set of the pins above against ``lib``; list what failed."""
    bad = list(golden_failures(lib))
    specs = [small_spec(201, H=4, Hkv=2, d=16, n_req=4, window=0, max_s=90),
             small_spec(202, H=8, Hkv=2, d=16, n_req=4, window=7, max_s=90),
             small_spec(203, H=4, Hkv=2, d=16, n_req=4, kv_dtype=1, max_s=90)]
    for sp in specs:
        case = W.make_case(sp)
        try:
            out, lse = run_oracle(case, lib=lib)
        except oracle.OracleError:
            bad.append(sp.name + ":error")
            continue
        ob, lb = run_brute(case)
        if rel_err(out, ob) > 1e-12 or rel_err(lse, lb) > 1e-12:
            bad.append(sp.name + ":brute")
        try:
            out2, lse2 = run_oracle(case, lib=lib, num_splits=3)
            if rel_err(out2, out) > 1e-12 or rel_err(lse2, lse) > 1e-12:
                bad.append(sp.name + ":split")
        except oracle.OracleError:
            bad.append(sp.name + ":split-error")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(int(c), lib=lib) for c in codes])
    if not np.all((np.isnan(ref) & np.isnan(got)) | (ref == got)):
        bad.append("e4m3")
    return bad


def test_pins_pass_on_the_oracle():
    assert pin_failures(None) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, tmp_path):
    src_path = os.path.join(os.path.dirname(HERE), "oracle", "pattn_ref.c")
    src = open(src_path).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "mut.c"
    so_path = tmp_path / "libmut.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                    str(so_path), str(c_path), "-lm"], check=True)
    lib = oracle.bind(str(so_path))
    assert pin_failures(lib), f"planted mistake {name} went unnoticed"
