"""GPU parity of cascade attention (pattn_cascade_fwd): batches whose
requests share their first common_prefix_len keys (the same blocks in every
block-table row) must give plain attention -- the float64 oracle's result --
and pattn_varlen_fwd's result within the tolerance.  Decode-only and mixed
batches, short and long prefixes, f16, e4m3 caches (the prefix pass then runs
the tensor-core prefill over widened e4m3 tiles), and a request whose cached
context does not cover the prefix (reported as bad metadata, others exact)."""
import numpy as np
import pytest
import torch

import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from gpu_util import assert_close, oracle_all, run_gpu

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_varlen_attention_attn_gb300 import _build
    _build.build()
    pa.load()


def shared_prefix_case(name, q_lens, seq_lens, H, Hkv, d, bs, prefix, seed, kv_dtype=0):
    spec = W.CaseSpec(name, q_lens, seq_lens, H, Hkv, d, bs,
                      pool_blocks=sum((s + bs - 1) // bs for s in seq_lens) + 4, seed=seed,
                      kv_dtype=kv_dtype)
    case = W.make_case(spec, device=DEV)
    n = prefix // bs
    case.block_table[:, :n] = case.block_table[0, :n].clone()
    return case


def run_cascade(case, prefix, num_splits=0):
    s = case.spec
    out = torch.full_like(case.q, float("nan"))
    pa.cascade_forward(case.q, case.kv_cache, case.block_table, case.seq_lens,
                       case.query_start_loc, scale=case.scale, num_heads=s.num_heads,
                       num_kv_heads=s.num_kv_heads, head_size=s.head_size,
                       block_size=s.block_size, common_prefix_len=prefix, kv_dtype=s.kv_dtype,
                       kv_scale=case.kv_scale if s.kv_dtype == W.KV_FP8_E4M3 else None,
                       max_query_len=case.max_query_len, max_seq_len=case.max_seq_len,
                       num_splits=num_splits, out=out)
    st = pa.pattn_read_device_status(pa.forward.last_ext)
    torch.cuda.synchronize()
    return out, st


def _rows(case):
    qsl = case.query_start_loc.cpu().numpy()
    return int(qsl[0]), int(qsl[-1])


@pytest.mark.parametrize("prefix,G,d", [(16, 4, 128), (512, 8, 128), (1024, 4, 64)])
def test_cascade_decode_batch(prefix, G, d):
    rng = np.random.default_rng(prefix + G)
    B, Hkv, bs = 12, 2, 16
    seq = [prefix + int(x) for x in rng.integers(1, 700, B)]
    case = shared_prefix_case("casc_dec", [1] * B, seq, G * Hkv, Hkv, d, bs, prefix, 1800 + prefix)
    ref, _ = oracle_all(case)
    out, st = run_cascade(case, prefix)
    assert st == 0
    a, b = _rows(case)
    assert_close(out[a:b].float().cpu().numpy(), ref[a:b], 0)
    plain = run_gpu(case)
    assert_close(out[a:b].float().cpu().numpy(), plain[a:b].float().cpu().numpy(), 0)


@pytest.mark.parametrize("bs", [16, 64])
@pytest.mark.parametrize("splits", [0, 3])
def test_cascade_mixed_batch(bs, splits):
    prefix = 256
    q_lens = [200, 1, 1, 64, 1, 130]
    seq_lens = [prefix + 300, prefix + 900, prefix + 5, prefix + 64, prefix + 2000, prefix + 130]
    case = shared_prefix_case("casc_mix", q_lens, seq_lens, 8, 2, 128, bs, prefix, 1900 + bs)
    ref, _ = oracle_all(case)
    out, st = run_cascade(case, prefix, num_splits=splits)
    assert st == 0
    a, b = _rows(case)
    assert_close(out[a:b].float().cpu().numpy(), ref[a:b], 0)


def test_cascade_f16():
    prefix = 128
    case = shared_prefix_case("casc_f16", [1, 50, 1, 1], [400, 300, 129, 700], 16, 4, 128, 16,
                              prefix, 1950, kv_dtype=W.KV_F16)
    ref, _ = oracle_all(case)
    out, st = run_cascade(case, prefix)
    assert st == 0
    a, b = _rows(case)
    assert_close(out[a:b].float().cpu().numpy(), ref[a:b], W.KV_F16)


@pytest.mark.parametrize("bs", [16, 128])
def test_cascade_e4m3_mixed_batch(bs):
    prefix = 256
    q_lens = [200, 1, 1, 64, 1, 130]
    seq_lens = [prefix + 300, prefix + 900, prefix + 5, prefix + 64, prefix + 2000, prefix + 130]
    case = shared_prefix_case("casc_e4m3", q_lens, seq_lens, 8, 2, 128, bs, prefix, 1990 + bs,
                              kv_dtype=W.KV_FP8_E4M3)
    ref, _ = oracle_all(case)
    out, st = run_cascade(case, prefix)
    assert st == 0
    a, b = _rows(case)
    assert_close(out[a:b].float().cpu().numpy(), ref[a:b], W.KV_FP8_E4M3)


@pytest.mark.parametrize("d", [64, 128])
def test_cascade_e4m3_decode_batch(d):
    rng = np.random.default_rng(d)
    B, Hkv, G, bs, prefix = 10, 2, 4, 16, 512
    seq = [prefix + int(x) for x in rng.integers(1, 700, B)]
    case = shared_prefix_case("casc_e4m3_dec", [1] * B, seq, G * Hkv, Hkv, d, bs, prefix,
                              1995 + d, kv_dtype=W.KV_FP8_E4M3)
    ref, _ = oracle_all(case)
    out, st = run_cascade(case, prefix)
    assert st == 0
    a, b = _rows(case)
    assert_close(out[a:b].float().cpu().numpy(), ref[a:b], W.KV_FP8_E4M3)


def test_cascade_context_shorter_than_prefix_is_reported():
    prefix = 64
    case = shared_prefix_case("casc_bad", [1, 40, 1], [300, 90, 200], 8, 2, 128, 16, prefix, 1970)
    # request 1: context 50 < prefix 64
    ref, _ = oracle_all(case)
    out, st = run_cascade(case, prefix)
    assert st == 5  # PATTN_ERR_BAD_METADATA
    assert torch.isfinite(out[_rows(case)[0]:_rows(case)[1]]).all()
    qsl = case.query_start_loc.cpu().numpy()
    for r in (0, 2):
        a, b = int(qsl[r]), int(qsl[r + 1])
        assert_close(out[a:b].float().cpu().numpy(), ref[a:b], 0)
