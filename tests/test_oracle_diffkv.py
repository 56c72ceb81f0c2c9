"""Pins of the oracle's DiffKV layout (CPU only).

"[vLLM] other attention backends", FlashAttention DiffKV: V may have its own
head size (head_size_v) and the cache is then asymmetric; the page gives no
shape.  The reading: one tensor [num_blocks][block_size][num_kv_heads]
[head_size + head_size_v], each row the token's K then its V.  Pinned by:
  - with head_size_v == head_size, the result equals the standard-layout
    result on a cache holding the same K and V (exactly);
  - the dense brute force (tests/brute.py), which slices K and V out of the
    de-paged rows, for head sizes that differ both ways;
  - a one-key window: every row's output is exactly that key's V part;
  - split == unsplit.
Planted mistakes in the oracle's DiffKV indexing must each fail one of them."""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from brute import brute_attention
from cases import case_args, diffkv_case

HERE = os.path.dirname(os.path.abspath(__file__))


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    ok = ~np.isnan(b)
    if np.isnan(a[ok]).any():
        return math.inf
    return float(np.max(np.abs(a[ok] - b[ok])) / max(1.0, np.max(np.abs(b[ok]))))


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _oracle(dc, lib=None, **over):
    c = dc.case
    kw = case_args(c)
    kw.update(over)
    return oracle.ref_varlen(_bits(c.q), _bits(dc.cache), c.block_table.cpu().numpy(),
                             c.seq_lens.cpu().numpy(), c.query_start_loc.cpu().numpy(),
                             head_size_v=dc.dv, lib=lib, **kw)


def diffkv_failures(lib):
    bad = []
    # same head sizes: the standard layout holding the same K and V
    dc = diffkv_case(501, H=4, Hkv=2, dk=32, dv=32, n_req=4, max_s=80)
    c = dc.case
    std = torch.stack([dc.cache[..., :32], dc.cache[..., 32:]]).contiguous()
    try:
        a = _oracle(dc, lib=lib)
        b = oracle.ref_varlen(_bits(c.q), _bits(std), c.block_table.cpu().numpy(),
                              c.seq_lens.cpu().numpy(), c.query_start_loc.cpu().numpy(),
                              lib=lib, **case_args(c))
        if not (np.array_equal(a[0], b[0], equal_nan=True) and
                np.array_equal(a[1], b[1], equal_nan=True)):
            bad.append("same-size")
    except oracle.OracleError:
        bad.append("same-size:error")
    # different head sizes, both ways: brute force and split == unsplit
    for seed, dk, dv, window in ((502, 32, 64, 0), (503, 64, 32, 0), (504, 32, 96, 11)):
        dc = diffkv_case(seed, H=4, Hkv=2, dk=dk, dv=dv, n_req=4, max_s=80, window=window)
        try:
            out, lse = _oracle(dc, lib=lib)
            out3, lse3 = _oracle(dc, lib=lib, num_splits=3)
        except oracle.OracleError:
            bad.append(f"{seed}:error")
            continue
        c = dc.case
        ob, lb = brute_attention(c.q, dc.cache, c.block_table, c.seq_lens, c.query_start_loc,
                                 head_size_v=dv, **case_args(c))
        if out.shape[-1] != dv or _rel(out, ob) > 1e-12 or _rel(lse, lb) > 1e-12:
            bad.append(f"{seed}:brute")
        if _rel(out3, out) > 1e-12 or _rel(lse3, lse) > 1e-12:
            bad.append(f"{seed}:split")
    # a one-key window: out is the V part of the row's own key, exactly
    dc = diffkv_case(505, H=2, Hkv=1, dk=32, dv=64, n_req=3, max_s=60, window=1)
    try:
        out, _ = _oracle(dc, lib=lib)
    except oracle.OracleError:
        return bad + ["window1:error"]
    c = dc.case
    cache = dc.cache.float().double().numpy()
    bt = c.block_table.cpu().numpy()
    qsl = c.query_start_loc.cpu().numpy()
    for r, (ql, s) in enumerate(zip(c.spec.q_lens, c.spec.seq_lens)):
        for i in range(ql):
            k = s - ql + i
            v = cache[bt[r, k // 16], k % 16, 0, 32:]
            if not np.array_equal(out[qsl[r] + i, 0], v):
                bad.append("window1")
    return bad


def test_diffkv_pins_pass_on_the_oracle():
    assert diffkv_failures(None) == []


MUTATIONS = {
    "k_and_v_parts_swapped": ("(kv_index ? jb->head_size + j : j)",
                              "(kv_index ? j : jb->head_size_v + j)"),
    "v_offset_by_v_size": ("(kv_index ? jb->head_size + j : j)",
                           "(kv_index ? jb->head_size_v + j : j)"),
    "row_stride_doubled_k": ("(jb->head_size + jb->head_size_v) + (kv_index",
                             "(2 * jb->head_size) + (kv_index"),
    "v_read_at_k_width": ("for (int j = 0; j < dv; ++j) o[j] += w * cache_elem(jb, 1, blk, slot, g, j);",
                          "for (int j = 0; j < d && j < dv; ++j) o[j] += w * cache_elem(jb, 1, blk, slot, g, j);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_diffkv_mistakes_are_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "pattn_ref.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
    (tmp_path / "mut.c").write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(tmp_path / "mut.c"), "-lm"], check=True)
    lib = oracle.bind(str(so))
    assert diffkv_failures(lib), f"{name} went unnoticed"
