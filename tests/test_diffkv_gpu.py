"""GPU parity of attention over a DiffKV cache (pattn_ext_t.head_size_v > 0:
[num_blocks, block_size, num_kv_heads, head_size + head_size_v], each row K
then V) against the float64 oracle on the same seeded inputs: head sizes that
differ both ways and up to 256, GQA ratios 1, 3, 4 and 16, mixed prefill /
chunk / decode batches spanning several 32-key tiles with ragged tails, a
sliding window, f16, attention sinks, equal head sizes, and a block id
outside the pool (reported, rows finite, other requests exact)."""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from cases import case_args, diffkv_case
from gpu_util import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_varlen_attention_attn_gb300 import _build
    _build.build()
    pa.load()


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _gpu(dc, sinks=None, expect=0):
    c, s = dc.case, dc.case.spec
    out = torch.full((c.q.shape[0], s.num_heads, dc.dv), float("nan"), dtype=c.q.dtype,
                     device=DEV)
    pa.forward(c.q, dc.cache, c.block_table, c.seq_lens, c.query_start_loc, scale=c.scale,
               num_heads=s.num_heads, num_kv_heads=s.num_kv_heads, head_size=s.head_size,
               block_size=s.block_size, window=s.window, causal=s.causal, kv_dtype=s.kv_dtype,
               max_query_len=c.max_query_len, max_seq_len=c.max_seq_len, out=out,
               sinks=sinks, head_size_v=dc.dv)
    st = pa.pattn_read_device_status(pa.forward.last_ext)
    torch.cuda.synchronize()
    assert st == expect, pa.pattn_status_string(st)
    return out


def _oracle(dc, sinks=None):
    c = dc.case
    return oracle.ref_varlen(_bits(c.q), _bits(dc.cache), c.block_table.cpu().numpy(),
                             c.seq_lens.cpu().numpy(), c.query_start_loc.cpu().numpy(),
                             head_size_v=dc.dv,
                             sinks=None if sinks is None else sinks.cpu().numpy(),
                             **case_args(c))


def _rows(dc):
    qsl = dc.case.query_start_loc.cpu().numpy()
    return int(qsl[0]), int(qsl[-1])


@pytest.mark.parametrize("dk,dv,H,Hkv", [(128, 64, 8, 2), (64, 128, 6, 2), (192, 128, 16, 1),
                                         (96, 256, 4, 4), (32, 32, 16, 4)])
def test_matches_the_oracle(dk, dv, H, Hkv):
    dc = diffkv_case(1600 + dk + dv + H, H=H, Hkv=Hkv, dk=dk, dv=dv, n_req=5, max_s=420,
                     device=DEV)
    ref, _ = _oracle(dc)
    a, b = _rows(dc)
    assert_close(_gpu(dc)[a:b].float().cpu().numpy(), ref[a:b], W.KV_BF16)


@pytest.mark.parametrize("window,kv_dtype", [(0, W.KV_BF16), (700, W.KV_BF16), (0, W.KV_F16)])
def test_long_decode_rows_on_the_tensor_core_kernel(window, kv_dtype):
    # decode rows long enough to wrap the decode kernel's stage ring many
    # times, at the K 192 / V 128 shape, with and without a window
    dc = diffkv_case(1680 + window + kv_dtype, H=32, Hkv=8, dk=192, dv=128, n_req=12,
                     max_s=3000, window=window, kv_dtype=kv_dtype, kinds=("decode",),
                     device=DEV)
    ref, _ = _oracle(dc)
    a, b = _rows(dc)
    assert_close(_gpu(dc)[a:b].float().cpu().numpy(), ref[a:b], W.KV_BF16)


def test_window_sinks_and_f16():
    dc = diffkv_case(1650, H=8, Hkv=2, dk=128, dv=64, n_req=5, max_s=500, window=77,
                     kv_dtype=W.KV_F16, device=DEV)
    sinks = torch.tensor([0.5, -1.0, 3.0, -float("inf"), 2.0, 0.0, 8.0, -2.5],
                         dtype=torch.float32, device=DEV)
    ref, _ = _oracle(dc, sinks)
    a, b = _rows(dc)
    assert_close(_gpu(dc, sinks)[a:b].float().cpu().numpy(), ref[a:b], W.KV_F16)


def test_decode_batch_with_block_size_64():
    dc = diffkv_case(1660, H=8, Hkv=2, dk=128, dv=64, bs=64, n_req=8, max_s=900,
                     kinds=("decode",), device=DEV)
    ref, _ = _oracle(dc)
    a, b = _rows(dc)
    assert_close(_gpu(dc)[a:b].float().cpu().numpy(), ref[a:b], W.KV_BF16)


def test_block_id_outside_the_pool():
    dc = diffkv_case(1670, H=4, Hkv=2, dk=64, dv=128, n_req=4, max_s=300, device=DEV)
    ref, _ = _oracle(dc)
    nb = dc.cache.shape[0]
    dc.case.block_table[1, 0] = nb + 5
    out = _gpu(dc, expect=5)
    qsl = dc.case.query_start_loc.cpu().numpy()
    assert torch.isfinite(out[int(qsl[1]):int(qsl[2])]).all()
    for r in (0, 2, 3):
        a, b = int(qsl[r]), int(qsl[r + 1])
        if b > a:
            assert_close(out[a:b].float().cpu().numpy(), ref[a:b], W.KV_BF16)


@pytest.mark.parametrize("dk,dv,bs,kv_dtype", [(128, 64, 16, W.KV_BF16), (96, 256, 64, W.KV_F16),
                                               (64, 128, 32, W.KV_BF16)])
def test_cache_write_matches_the_oracle_bit_for_bit(dk, dv, bs, kv_dtype):
    T, Hkv, nb = 203, 3, 30
    g = torch.Generator().manual_seed(1700 + dk + dv + bs)
    dt = torch.float16 if kv_dtype == W.KV_F16 else torch.bfloat16
    key = torch.randn(T, Hkv, dk, generator=g).to(dt)
    value = torch.randn(T, Hkv, dv, generator=g).to(dt)
    cache = torch.randint(-(1 << 15), 1 << 15, (nb, bs, Hkv, dk + dv), generator=g,
                          dtype=torch.int32).to(torch.int16).view(dt)
    slots = torch.randperm(nb * bs, generator=g)[:T].to(torch.int64)
    slots[::7] = -1
    ref = oracle.reshape_and_cache_diffkv(_bits(key), _bits(value), _bits(cache).copy(),
                                          slots.numpy(), num_kv_heads=Hkv, head_size=dk,
                                          head_size_v=dv, block_size=bs)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = cache.to(DEV)
    pa.reshape_and_cache_diffkv(key.to(DEV), value.to(DEV), got, slots.to(DEV), block_size=bs,
                                kv_dtype=kv_dtype, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(_bits(got), ref)
    # a slot past the pool is reported and writes nothing
    slots2 = slots.clone()
    slots2[3] = nb * bs + 1
    before = got.clone()
    pa.reshape_and_cache_diffkv(key[3:4].to(DEV), value[3:4].to(DEV), got, slots2[3:4].to(DEV),
                                block_size=bs, kv_dtype=kv_dtype, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert np.array_equal(_bits(got), _bits(before))  # bits: the cache holds NaN patterns


def test_attention_over_a_cache_filled_by_the_kernel():
    dc = diffkv_case(1710, H=8, Hkv=2, dk=128, dv=64, n_req=4, max_s=300, device=DEV)
    c = dc.case
    bt = c.block_table.cpu()
    toks = [(r, k) for r, s in enumerate(c.spec.seq_lens) for k in range(s)]
    slots = torch.tensor([int(bt[r, k // 16]) * 16 + k % 16 for r, k in toks], dtype=torch.int64)
    rows = dc.cache.reshape(-1, 2, 192)[slots.to(DEV)]
    ref, _ = _oracle(dc)
    dc.cache.zero_()
    pa.reshape_and_cache_diffkv(rows[:, :, :128].contiguous(), rows[:, :, 128:].contiguous(),
                                dc.cache, slots.to(DEV), block_size=16)
    a, b = _rows(dc)
    assert_close(_gpu(dc)[a:b].float().cpu().numpy(), ref[a:b], W.KV_BF16)
