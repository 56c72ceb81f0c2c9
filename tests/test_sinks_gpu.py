"""GPU parity of attention sinks (pattn_ext_t.sinks) against the float64
oracle given the same per-head logits: decode rows in one partition and in
several (the sink enters the in-kernel merge), prefill rows with both
sub-tile pairings (even and odd GQA group size) and a sliding window, mixed
batches, f16 and e4m3 caches, cascade (the sink enters its final merge once),
a dominant sink (rows near 0), and a sink of -inf, which must give exactly the
output of a call without sinks."""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from cases import small_spec
from gpu_util import _host, assert_close, oracle_kwargs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_varlen_attention_attn_gb300 import _build
    _build.build()
    pa.load()


def _sinks(H, seed, shift=0.0):
    rng = np.random.default_rng(seed)
    s = (rng.normal(0.0, 2.0, H) + shift).astype(np.float32)
    return torch.from_numpy(s).to(DEV)


def _gpu(case, sinks, num_splits=0):
    s = case.spec
    out = torch.full_like(case.q, float("nan"))
    pa.forward(case.q, case.kv_cache, case.block_table, case.seq_lens, case.query_start_loc,
               scale=case.scale, num_heads=s.num_heads, num_kv_heads=s.num_kv_heads,
               head_size=s.head_size, block_size=s.block_size, window=s.window,
               causal=s.causal, kv_dtype=s.kv_dtype,
               kv_scale=case.kv_scale if s.kv_dtype == W.KV_FP8_E4M3 else None,
               max_query_len=case.max_query_len, max_seq_len=case.max_seq_len,
               num_splits=num_splits, out=out, sinks=sinks)
    st = pa.pattn_read_device_status(pa.forward.last_ext)
    torch.cuda.synchronize()
    assert st == 0, pa.pattn_status_string(st)
    return out


def _oracle(case, sinks):
    q, kv, bt, sl, qsl = _host(case)
    return oracle.ref_varlen(q, kv, bt, sl, qsl, sinks=sinks.cpu().numpy(),
                             **oracle_kwargs(case))


def _check(case, out, sinks):
    ref, _ = _oracle(case, sinks)
    qsl = case.query_start_loc.cpu().numpy()
    a, b = int(qsl[0]), int(qsl[-1])
    return assert_close(out[a:b].float().cpu().numpy(), ref[a:b], case.spec.kv_dtype)


@pytest.mark.parametrize("splits", [1, 3, 0])
@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_FP8_E4M3])
def test_decode_rows(splits, kv_dtype):
    sp = small_spec(1400 + splits + 10 * kv_dtype, H=8, Hkv=2, d=128, bs=16, n_req=6,
                    max_s=900, kinds=("decode",), kv_dtype=kv_dtype)
    case = W.make_case(sp, device=DEV)
    sinks = _sinks(8, sp.seed)
    _check(case, _gpu(case, sinks, num_splits=splits), sinks)


@pytest.mark.parametrize("H,Hkv,window", [(8, 2, 0), (6, 2, 0), (8, 2, 150)])
def test_prefill_and_mixed_rows(H, Hkv, window):
    sp = small_spec(1420 + H + window, H=H, Hkv=Hkv, d=128, bs=16, n_req=5, max_s=700,
                    window=window)
    case = W.make_case(sp, device=DEV)
    sinks = _sinks(H, sp.seed)
    _check(case, _gpu(case, sinks), sinks)


def test_f16_head_size_64():
    sp = small_spec(1440, H=4, Hkv=2, d=64, bs=32, n_req=5, max_s=600, kv_dtype=W.KV_F16)
    case = W.make_case(sp, device=DEV)
    sinks = _sinks(4, sp.seed)
    _check(case, _gpu(case, sinks, num_splits=2), sinks)


def test_dominant_sink_drives_rows_to_zero():
    sp = small_spec(1450, H=4, Hkv=2, d=128, bs=16, n_req=5, max_s=500)
    case = W.make_case(sp, device=DEV)
    sinks = torch.tensor([60.0, 200.0, 1e30, 3.0], dtype=torch.float32, device=DEV)
    out = _gpu(case, sinks, num_splits=2)
    _check(case, out, sinks)
    qsl = case.query_start_loc.cpu().numpy()
    rows = out[int(qsl[0]):int(qsl[-1])]
    assert torch.count_nonzero(rows[:, 1:3]) == 0  # weights underflow or the sum overflows


def test_minus_inf_sink_is_no_sink():
    sp = small_spec(1460, H=8, Hkv=2, d=128, bs=16, n_req=6, max_s=600)
    case = W.make_case(sp, device=DEV)
    none = _gpu(case, None, num_splits=3)
    minf = _gpu(case, torch.full((8,), -float("inf"), device=DEV), num_splits=3)
    assert torch.equal(none, minf)


def test_cascade():
    rng = np.random.default_rng(1470)
    B, H, Hkv, d, bs, prefix = 6, 8, 2, 128, 16, 256
    ql = [1, 1, 37, 1, 200, 1]
    # every request's cached context covers the prefix
    seq = [prefix + q + int(x) for q, x in zip(ql, rng.integers(0, 400, B))]
    spec = W.CaseSpec("sink_cascade", ql, seq, H, Hkv, d, bs,
                      pool_blocks=sum((s + bs - 1) // bs for s in seq) + 4, seed=1470)
    case = W.make_case(spec, device=DEV)
    case.block_table[:, :prefix // bs] = case.block_table[0, :prefix // bs].clone()
    sinks = _sinks(H, 1470)
    out = torch.full_like(case.q, float("nan"))
    pa.cascade_forward(case.q, case.kv_cache, case.block_table, case.seq_lens,
                       case.query_start_loc, scale=case.scale, num_heads=H, num_kv_heads=Hkv,
                       head_size=d, block_size=bs, common_prefix_len=prefix,
                       max_query_len=case.max_query_len, max_seq_len=case.max_seq_len,
                       out=out, sinks=sinks)
    st = pa.pattn_read_device_status(pa.forward.last_ext)
    torch.cuda.synchronize()
    assert st == 0, pa.pattn_status_string(st)
    _check(case, out, sinks)
