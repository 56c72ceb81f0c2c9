"""Pins of the oracle's f16 path (CPU only): the IEEE binary16 decoder against
numpy's float16 for all 65,536 patterns, and whole-batch attention with f16
q and cache against the dense brute force (whose conversions go through
torch's float16).  A planted mistake in the decoder must fail the pins."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads as W
from brute import brute_attention
from cases import case_args, host_arrays, small_spec

HERE = os.path.dirname(os.path.abspath(__file__))


def decoder_failures(lib):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(int(b), lib=lib) for b in bits])
    same = (np.isnan(ref) & np.isnan(got)) | (ref == got)
    return [] if same.all() else ["f16-decoder"]


def test_f16_decoder_all_patterns():
    assert decoder_failures(None) == []


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    m = np.isfinite(b)
    return float(np.max(np.abs(a[m] - b[m])) / max(1e-300, np.max(np.abs(b[m]))))


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("window", [0, 9])
def test_f16_attention_matches_brute_force(seed, window):
    spec = small_spec(1300 + seed + window, H=8, Hkv=2, d=16, bs=16, n_req=4, max_s=90,
                      window=window, kv_dtype=W.KV_F16)
    case = W.make_case(spec)
    q, kv, bt, sl, qsl = host_arrays(case)
    out, lse = oracle.ref_varlen(q, kv, bt, sl, qsl, **case_args(case))
    ob, lb = brute_attention(case.q, case.kv_cache, case.block_table, case.seq_lens,
                             case.query_start_loc, **case_args(case))
    a, b = int(qsl[0]), int(qsl[-1])
    assert _rel(out[a:b], ob[a:b]) <= 1e-12 and _rel(lse[a:b], lb[a:b]) <= 1e-12


MUTATIONS = {
    "f16_bias": ("mag = ldexp(1.0 + (double)m / 1024.0, e - 15);",
                 "mag = ldexp(1.0 + (double)m / 1024.0, e - 14);"),
    "f16_subnormal": ("mag = ldexp((double)m, -24);", "mag = ldexp((double)m, -23);"),
    "q_decoded_as_bf16": ("qv[j] = jb->kv_dtype == 2 ? pattn_ref_f16_to_double(bits) : pattn_ref_bf16_to_double(bits);",
                          "qv[j] = pattn_ref_bf16_to_double(bits);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "pattn_ref.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
    (tmp_path / "mut.c").write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(tmp_path / "mut.c"), "-lm"], check=True)
    lib = oracle.bind(str(so))
    bad = decoder_failures(lib)
    spec = small_spec(1399, H=8, Hkv=2, d=16, bs=16, n_req=3, max_s=60, kv_dtype=W.KV_F16)
    case = W.make_case(spec)
    q, kv, bt, sl, qsl = host_arrays(case)
    out, _ = oracle.ref_varlen(q, kv, bt, sl, qsl, lib=lib, **case_args(case))
    ob, _ = brute_attention(case.q, case.kv_cache, case.block_table, case.seq_lens,
                            case.query_start_loc, **case_args(case))
    a, b = int(qsl[0]), int(qsl[-1])
    if _rel(out[a:b], ob[a:b]) > 1e-12:
        bad.append("brute")
    assert bad, f"{name} went unnoticed"
