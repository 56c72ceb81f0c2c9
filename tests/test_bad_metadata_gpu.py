"""Bad metadata on the GPU: block ids outside the pool, a query longer than its
sequence, a sequence longer than its block-table row, a longer query in a call
declared decode-only.  Each must be reported as PATTN_ERR_BAD_METADATA by
pattn_read_device_status, with no out-of-bounds access (block ids are clamped),
a finite output, zeroed rows where the request cannot be computed, and every
other request still exact.  The faults are made on the host, in the metadata;
no test makes the GPU fault."""
import numpy as np
import pytest
import torch

import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from cases import small_spec
from gpu_util import assert_close, oracle_all

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BAD = 5  # PATTN_ERR_BAD_METADATA


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_varlen_attention_attn_gb300 import _build
    _build.build()
    pa.load()


def _call(case, max_query_len=None, num_splits=0):
    s = case.spec
    out = torch.full_like(case.q, float("nan"))
    pa.forward(case.q, case.kv_cache, case.block_table, case.seq_lens, case.query_start_loc,
               scale=case.scale, num_heads=s.num_heads, num_kv_heads=s.num_kv_heads,
               head_size=s.head_size, block_size=s.block_size, window=s.window,
               causal=s.causal, kv_dtype=s.kv_dtype,
               kv_scale=case.kv_scale if s.kv_dtype else None,
               max_query_len=case.max_query_len if max_query_len is None else max_query_len,
               max_seq_len=case.max_seq_len, num_splits=num_splits, out=out)
    st = pa.pattn_read_device_status(pa.forward.last_ext)
    torch.cuda.synchronize()
    # reading the status clears it: a second read sees a clean word
    assert pa.pattn_read_device_status(pa.forward.last_ext) == 0
    return out, st


def _rows(case, r):
    qsl = case.query_start_loc.cpu().numpy()
    return int(qsl[r]), int(qsl[r + 1])


def _check_others(case, out, ref, bad_r):
    for r in range(len(case.spec.q_lens)):
        if r == bad_r:
            continue
        a, b = _rows(case, r)
        if b > a:
            assert_close(out[a:b].float().cpu().numpy(), ref[a:b], case.spec.kv_dtype)


@pytest.mark.parametrize("kind", ["decode", "prefill"])
@pytest.mark.parametrize("splits", [1, 3])
def test_block_id_outside_the_pool(kind, splits):
    spec = small_spec(900 + splits + (kind == "prefill"), H=8, Hkv=2, d=128, bs=16, n_req=4,
                      max_s=400, kinds=(kind,))
    case = W.make_case(spec, device=DEV)
    ref, _ = oracle_all(case)
    nb = case.kv_cache.shape[1]
    case.block_table[1, 0] = nb + 7
    case.block_table[1, 1] = -3
    out, st = _call(case, num_splits=splits)
    assert st == BAD
    assert torch.isfinite(out[slice(*_rows(case, 1))]).all()
    _check_others(case, out, ref, 1)


def test_query_longer_than_its_sequence():
    spec = small_spec(910, H=4, Hkv=2, d=64, bs=16, n_req=3, max_s=300, kinds=("prefill",))
    case = W.make_case(spec, device=DEV)
    ref, _ = oracle_all(case)
    a, b = _rows(case, 1)
    case.seq_lens[1] = (b - a) - 1
    out, st = _call(case)
    assert st == BAD
    assert torch.count_nonzero(out[a:b]) == 0
    _check_others(case, out, ref, 1)


@pytest.mark.parametrize("kind", ["decode", "prefill"])
def test_sequence_longer_than_its_block_table_row(kind):
    spec = small_spec(920 + (kind == "prefill"), H=8, Hkv=2, d=128, bs=16, n_req=3, max_s=300,
                      kinds=(kind,))
    case = W.make_case(spec, device=DEV)
    ref, _ = oracle_all(case)
    mbps = case.block_table.shape[1]
    case.seq_lens[2] = mbps * spec.block_size + 16
    out, st = _call(case)
    assert st == BAD
    a, b = _rows(case, 2)
    assert torch.count_nonzero(out[a:b]) == 0
    _check_others(case, out, ref, 2)


def test_longer_query_in_a_call_declared_decode_only():
    spec = W.CaseSpec("dec_only_bad", [1, 3, 1], [200, 150, 90], 8, 2, 128, 16,
                      pool_blocks=40, seed=930)
    case = W.make_case(spec, device=DEV)
    ref, _ = oracle_all(case)
    out, st = _call(case, max_query_len=1, num_splits=2)
    assert st == BAD
    a, b = _rows(case, 1)
    assert torch.count_nonzero(out[a:b]) == 0
    _check_others(case, out, ref, 1)
