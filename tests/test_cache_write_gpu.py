"""GPU parity of the KV-cache write (pattn_reshape_and_cache) against the
oracle's write, bit for bit over the whole cache: bf16 and e4m3 caches, head
sizes 64 and 128, block sizes 16 and 64, padding slots, values that saturate
e4m3, NaN inputs, and a slot past the pool (reported, nothing written).  The
last test fills a cache with the kernel and runs attention over it."""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from gpu_util import assert_close, oracle_all

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_varlen_attention_attn_gb300 import _build
    _build.build()
    pa.load()


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _cache_host(cache, kv_dtype):
    c = cache.detach().cpu()
    return c.view(torch.int16).numpy().view(np.uint16).copy() if kv_dtype == 0 else c.numpy().copy()


def _setup(seed, T, Hkv, d, bs, nb, kv_dtype, spread=3.0, pad_every=5):
    g = torch.Generator(device=DEV).manual_seed(seed)
    key = (torch.randn(T, Hkv, d, generator=g, device=DEV) * spread).to(torch.bfloat16)
    value = (torch.randn(T, Hkv, d, generator=g, device=DEV) * spread).to(torch.bfloat16)
    cg = torch.Generator().manual_seed(seed)
    slots = torch.randperm(nb * bs, generator=cg)[:T].to(torch.int64)
    if pad_every:
        slots[::pad_every] = -1
    if kv_dtype == 0:
        cache = torch.randint(-(1 << 15), 1 << 15, (2, nb, bs, Hkv, d), generator=cg,
                              dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    else:
        cache = torch.randint(0, 256, (2, nb, bs, Hkv, d), generator=cg, dtype=torch.int32).to(
            torch.uint8)
    return key, value, slots.to(DEV), cache.to(DEV)


@pytest.mark.parametrize("kv_dtype", [0, 1])
@pytest.mark.parametrize("d,bs", [(128, 16), (64, 64), (128, 64)])
def test_cache_write_matches_the_oracle_bit_for_bit(kv_dtype, d, bs):
    T, Hkv, nb = 301, 4, 40
    key, value, slots, cache = _setup(50 + d + bs + kv_dtype, T, Hkv, d, bs, nb, kv_dtype)
    scale = (float(key.float().abs().max()) / 448, float(value.float().abs().max()) / 448)
    ref = oracle.reshape_and_cache(_bits(key), _bits(value), _cache_host(cache, kv_dtype),
                                   slots.cpu().numpy(), num_kv_heads=Hkv, head_size=d,
                                   block_size=bs, kv_dtype=kv_dtype, kv_scale=scale)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache(key, value, cache, slots, block_size=bs, kv_dtype=kv_dtype,
                         kv_scale=scale if kv_dtype else None, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(_cache_host(cache, kv_dtype), ref)


def test_e4m3_saturation_and_nan_match_the_oracle():
    T, Hkv, d, bs, nb = 64, 2, 128, 16, 8
    key, value, slots, cache = _setup(77, T, Hkv, d, bs, nb, 1, spread=50.0, pad_every=0)
    key[3, 1, 5] = float("nan")
    value[7, 0, 9] = float("inf")
    value[8, 1, 0] = -float("inf")
    scale = (0.05, 0.07)  # most |x| / scale exceed 448: saturated codes
    ref = oracle.reshape_and_cache(_bits(key), _bits(value), _cache_host(cache, 1),
                                   slots.cpu().numpy(), num_kv_heads=Hkv, head_size=d,
                                   block_size=bs, kv_dtype=1, kv_scale=scale)
    pa.reshape_and_cache(key, value, cache, slots, block_size=bs, kv_dtype=1, kv_scale=scale)
    torch.cuda.synchronize()
    got = _cache_host(cache, 1)
    assert np.array_equal(got, ref)
    assert (got == 0x7E).sum() > 1000 and (got == 0xFE).sum() > 1000


def test_slot_past_the_pool_is_reported_and_not_written():
    T, Hkv, d, bs, nb = 40, 2, 64, 16, 6
    key, value, slots, cache = _setup(88, T, Hkv, d, bs, nb, 0)
    before = _cache_host(cache, 0)
    slots_h = slots.cpu()
    slots_h[11] = nb * bs + 3
    ref = before.copy()
    good = slots_h.clone()
    good[11] = -1
    oracle.reshape_and_cache(_bits(key), _bits(value), ref, good.numpy(), num_kv_heads=Hkv,
                             head_size=d, block_size=bs)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache(key, value, cache, slots_h.to(DEV), block_size=bs, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert np.array_equal(_cache_host(cache, 0), ref)


def test_attention_over_a_cache_filled_by_the_kernel():
    """Decode step: every request's keys 0 .. s-1 are written by the cache
    write (slots from the request's block table), then attention runs."""
    spec = W.CaseSpec("cw_decode", [1, 1, 1, 1], [37, 300, 129, 512], 16, 2, 128, 16,
                      pool_blocks=80, seed=1201)
    case = W.make_case(spec, device=DEV)
    bt = case.block_table.cpu()
    tok_slots, rows = [], []
    for r, s in enumerate(spec.seq_lens):
        for k in range(s):
            tok_slots.append(int(bt[r, k // 16]) * 16 + k % 16)
            rows.append((r, k))
    kv_host = case.kv_cache.cpu()
    key = torch.stack([kv_host[0, sl // 16, sl % 16] for sl in tok_slots]).to(DEV)
    value = torch.stack([kv_host[1, sl // 16, sl % 16] for sl in tok_slots]).to(DEV)
    ref, _ = oracle_all(case)
    case.kv_cache.zero_()
    pa.reshape_and_cache(key, value, case.kv_cache,
                         torch.tensor(tok_slots, dtype=torch.int64, device=DEV), block_size=16)
    out = torch.zeros_like(case.q)
    pa.forward(case.q, case.kv_cache, case.block_table, case.seq_lens, case.query_start_loc,
               scale=case.scale, num_heads=16, num_kv_heads=2, head_size=128, block_size=16,
               max_query_len=1, max_seq_len=512, out=out)
    torch.cuda.synchronize()
    assert_close(out.float().cpu().numpy(), ref, 0)
