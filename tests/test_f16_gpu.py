"""GPU parity with f16 q, cache and output (PATTN_KV_F16) against the float64
oracle: decode at several group sizes, head sizes and partition counts,
prefill at several block sizes, mixed batches with a window, a larger decode
batch, the workspace-free decode entry point's kernels, and the cache write
(a 16-bit copy).  Tolerance: the bf16 one (f16 carries more mantissa)."""
import numpy as np
import pytest
import torch

import oracle
import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from cases import small_spec
from gpu_util import check_case

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
F16 = W.KV_F16


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_varlen_attention_attn_gb300 import _build
    _build.build()
    pa.load()


def make(spec):
    return W.make_case(spec, device=DEV)


@pytest.mark.parametrize("G,Hkv", [(1, 4), (4, 2), (8, 8), (16, 1)])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("splits", [1, 3])
def test_f16_decode(G, Hkv, D, splits):
    spec = small_spec(1400 + G + Hkv + D + splits, H=G * Hkv, Hkv=Hkv, d=D, bs=16, n_req=4,
                      max_s=600, kv_dtype=F16, kinds=("decode",))
    check_case(make(spec), num_splits=splits)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 64, 256])
def test_f16_prefill(D, bs):
    spec = small_spec(1500 + D + bs, H=4, Hkv=2, d=D, bs=bs, n_req=3, max_s=400,
                      kv_dtype=F16, kinds=("prefill", "chunk"))
    check_case(make(spec))


@pytest.mark.parametrize("window", [0, 33])
def test_f16_mixed_batch(window):
    spec = small_spec(1600 + window, H=8, Hkv=2, d=128, bs=16, n_req=8, max_s=700,
                      window=window, kv_dtype=F16)
    check_case(make(spec))


def test_f16_larger_decode_batch():
    spec = W.CaseSpec("f16_decode_gqa", [1] * 24,
                      [int(x) for x in np.random.default_rng(5).integers(512, 4096, 24)],
                      32, 8, 128, 16, pool_blocks=7000, seed=1701, kv_dtype=F16)
    check_case(make(spec))


def test_f16_cache_write_is_a_copy():
    g = torch.Generator(device=DEV).manual_seed(3)
    key = torch.randn(50, 2, 128, generator=g, device=DEV).to(torch.float16)
    value = torch.randn(50, 2, 128, generator=g, device=DEV).to(torch.float16)
    cache = torch.zeros(2, 8, 16, 2, 128, dtype=torch.float16, device=DEV)
    slots = torch.randperm(128, generator=torch.Generator().manual_seed(3))[:50].to(DEV)
    slots[::7] = -1
    pa.reshape_and_cache(key, value, cache, slots, block_size=16, kv_dtype=F16)
    ref = oracle.reshape_and_cache(
        key.cpu().view(torch.int16).numpy().view(np.uint16),
        value.cpu().view(torch.int16).numpy().view(np.uint16),
        np.zeros((2, 8, 16, 2, 128), dtype=np.uint16), slots.cpu().numpy(), num_kv_heads=2,
        head_size=128, block_size=16, kv_dtype=F16)
    torch.cuda.synchronize()
    assert np.array_equal(cache.cpu().view(torch.int16).numpy().view(np.uint16), ref)
