"""Bounded waits on the GPU: a wait that runs out is reported, not a hang.

Every mbarrier wait in the kernels gives up after a time limit, records
PATTN_ERR_DEVICE_TIMEOUT in the workspace status word, and unwinds: the other
roles of the CTA see an abort flag, the producers wait (bounded) for the
copies they armed, the MMA thread waits for its MMAs, and the CTA frees its
TMEM and exits.  These tests reach that path without faulting or hanging
anything: they load the wait-test build of the library (the same sources
compiled with PATTN_WAIT_TEST: a 10 ms limit, and a hook by which CTA 0 posts
no bytes and issues no copy for its first K tile or decode unit, a barrier
phase that nothing then completes).  The call must report the timeout and
leave finite output, and the next call in the same context, with the hook
off, must match the float64 oracle: the prefill kernel, which holds TMEM,
would otherwise block on its TMEM allocation.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from cases import small_spec
from gpu_util import assert_close, oracle_all, valid_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TIMEOUT = 6  # PATTN_ERR_DEVICE_TIMEOUT


@pytest.fixture(scope="module")
def wlib():
    from paged_varlen_attention_attn_gb300 import _build
    lib = pa.load(_build.build_wait_test())
    lib.pattn_test_set_wait_skip.argtypes = [ctypes.c_int]
    lib.pattn_test_set_wait_skip.restype = None
    lib.pattn_test_set_wait_skip(0)
    yield lib
    lib.pattn_test_set_wait_skip(0)


def run(lib, case, out):
    s = case.spec
    pa.forward(case.q, case.kv_cache, case.block_table, case.seq_lens, case.query_start_loc,
               scale=case.scale, num_heads=s.num_heads, num_kv_heads=s.num_kv_heads,
               head_size=s.head_size, block_size=s.block_size, window=s.window,
               causal=s.causal, kv_dtype=s.kv_dtype,
               kv_scale=case.kv_scale if s.kv_dtype else None,
               max_query_len=case.max_query_len, max_seq_len=case.max_seq_len,
               num_splits=s.num_splits, out=out, lib=lib)
    return pa.pattn_read_device_status(pa.forward.last_ext, lib=lib)


CASES = {
    # skip 1: the prefill kernel's first K tile on CTA 0 (prefill rows only)
    1: dict(seed=5151, H=8, Hkv=2, d=128, bs=16, n_req=4, max_s=700, kinds=("prefill",)),
    # skip 2: the decode kernel's first unit on CTA 0 (decode rows only)
    2: dict(seed=5252, H=16, Hkv=2, d=128, bs=16, n_req=6, max_s=2000, kinds=("decode",)),
}


@pytest.mark.parametrize("mode", [1, 2])
def test_wait_that_runs_out_is_reported_and_the_next_call_is_correct(wlib, mode):
    kw = dict(CASES[mode])
    case = W.make_case(small_spec(kw.pop("seed"), **kw), device=DEV)
    out = torch.zeros_like(case.q)
    wlib.pattn_test_set_wait_skip(mode)
    try:
        st = run(wlib, case, out)
    finally:
        wlib.pattn_test_set_wait_skip(0)
    torch.cuda.synchronize()
    assert st == TIMEOUT, pa.pattn_status_string(st, lib=wlib)
    assert torch.isfinite(out.float()).all()

    # the same context, the hook off: every CTA's result is right again
    out2 = torch.full_like(case.q, float("nan"))
    st = run(wlib, case, out2)
    torch.cuda.synchronize()
    assert st == 0, pa.pattn_status_string(st, lib=wlib)
    ref, _ = oracle_all(case)
    a, b = valid_rows(case)
    assert_close(out2[a:b].float().cpu().numpy(), ref[a:b], case.spec.kv_dtype)


def test_product_library_is_unaffected_after_a_timeout(wlib):
    # the product library in the same process still computes correct rows
    case = W.make_case(small_spec(5353, H=8, Hkv=2, d=128, bs=16, n_req=5, max_s=500),
                       device=DEV)
    out = torch.zeros_like(case.q)
    st = run(pa.load(), case, out)
    torch.cuda.synchronize()
    assert st == 0
    ref, _ = oracle_all(case)
    a, b = valid_rows(case)
    assert_close(out[a:b].float().cpu().numpy(), ref[a:b], case.spec.kv_dtype)
