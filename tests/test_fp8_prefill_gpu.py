"""GPU parity of e4m3 caches with prefill rows: the decode rows run on the
decode kernel and the prefill rows (full and chunked prefills) on the
tensor-core prefill kernel, which at head size 128 takes the K codes into
8-bit score MMAs against a split Q and widens V to f16 in shared memory (at
64 it widens both), and applies the per-tensor scales.  Compared with the
float64 oracle at the e4m3 tolerance: head sizes 64 and 128, even and odd GQA
ratios, a sliding window, block sizes 64, 128 and 256 (pages of a key tile or
more), attention sinks, a batch of chunked prefills beside many decodes, a
prefill request whose query is longer than its sequence (reported, rows zero,
others exact), and query rows whose magnitudes span 2^-40 to 2^8 (both head
sizes)."""
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


def _gpu(case, sinks=None, expect=0):
    s = case.spec
    out = torch.full_like(case.q, float("nan"))
    pa.forward(case.q, case.kv_cache, case.block_table, case.seq_lens, case.query_start_loc,
               scale=case.scale, num_heads=s.num_heads, num_kv_heads=s.num_kv_heads,
               head_size=s.head_size, block_size=s.block_size, window=s.window,
               causal=s.causal, kv_dtype=s.kv_dtype, kv_scale=case.kv_scale,
               max_query_len=case.max_query_len, max_seq_len=case.max_seq_len, out=out,
               sinks=sinks)
    st = pa.pattn_read_device_status(pa.forward.last_ext)
    torch.cuda.synchronize()
    assert st == expect, pa.pattn_status_string(st)
    return out


def _oracle(case, sinks=None):
    q, kv, bt, sl, qsl = _host(case)
    return oracle.ref_varlen(q, kv, bt, sl, qsl,
                             sinks=None if sinks is None else sinks.cpu().numpy(),
                             **oracle_kwargs(case))


def _check(case, out, sinks=None, skip=()):
    ref, _ = _oracle(case, sinks)
    qsl = case.query_start_loc.cpu().numpy()
    for r in range(len(case.spec.q_lens)):
        a, b = int(qsl[r]), int(qsl[r + 1])
        if b > a and r not in skip:
            assert_close(out[a:b].float().cpu().numpy(), ref[a:b], W.KV_FP8_E4M3)


@pytest.mark.parametrize("H,Hkv,d,bs,window", [(8, 2, 128, 16, 0), (6, 2, 64, 16, 0),
                                               (4, 4, 128, 64, 0), (16, 2, 128, 16, 90),
                                               (12, 4, 128, 256, 0), (8, 8, 64, 128, 0),
                                               (8, 2, 64, 16, 50), (6, 2, 128, 32, 130)])
def test_mixed_batches(H, Hkv, d, bs, window):
    sp = small_spec(1800 + H + d + bs + window, H=H, Hkv=Hkv, d=d, bs=bs, n_req=6, max_s=600,
                    window=window, kv_dtype=W.KV_FP8_E4M3)
    case = W.make_case(sp, device=DEV)
    _check(case, _gpu(case))


def test_sinks():
    sp = small_spec(1850, H=8, Hkv=2, d=128, n_req=5, max_s=500, kv_dtype=W.KV_FP8_E4M3)
    case = W.make_case(sp, device=DEV)
    sinks = torch.linspace(-3.0, 5.0, 8, dtype=torch.float32, device=DEV)
    _check(case, _gpu(case, sinks), sinks)


def test_chunked_prefills_beside_many_decodes():
    q_lens = [96, 130] + [1] * 20
    rng = np.random.default_rng(1860)
    seq = [400, 700] + [int(x) for x in rng.integers(100, 900, 20)]
    spec = W.CaseSpec("fp8_chunks", q_lens, seq, 16, 4, 128, 16,
                      pool_blocks=sum((s + 15) // 16 for s in seq) + 4, seed=1860,
                      kv_dtype=W.KV_FP8_E4M3)
    case = W.make_case(spec, device=DEV)
    _check(case, _gpu(case))


def test_query_longer_than_its_sequence():
    sp = small_spec(1870, H=4, Hkv=2, d=128, n_req=4, max_s=300, kinds=("prefill",),
                    kv_dtype=W.KV_FP8_E4M3)
    case = W.make_case(sp, device=DEV)
    qsl = case.query_start_loc.cpu().numpy()
    a, b = int(qsl[1]), int(qsl[2])
    ref, _ = _oracle(case)
    case.seq_lens[1] = (b - a) - 1
    out = _gpu(case, expect=5)
    assert torch.count_nonzero(out[a:b]) == 0
    for r in (0, 2, 3):
        x, y = int(qsl[r]), int(qsl[r + 1])
        if y > x:
            assert_close(out[x:y].float().cpu().numpy(), ref[x:y], W.KV_FP8_E4M3)


@pytest.mark.parametrize("d", [128, 64])
def test_query_rows_of_very_different_magnitudes(d):
    # At head size 128 the scores are 8-bit MMAs on the K codes against a Q
    # split per row into e4m3 hi + lo codes after a power-of-two scaling; at
    # 64 Q rows are scaled by a power of two into f16's range for the f16
    # MMAs.  Rows scaled from 2^-40 to 2^8 (and rows with one large entry
    # among small ones) must still match the definition.  (Larger rows would
    # give scores whose log2-domain magnitude, above ~2^20, an fp32 softmax
    # cannot resolve to a unit: a limit of every path, not of the scaling.)
    sp = small_spec(1880 + d, H=8, Hkv=2, d=d, bs=16, n_req=4, max_s=400, kinds=("prefill",),
                    kv_dtype=W.KV_FP8_E4M3)
    case = W.make_case(sp, device=DEV)
    T, H, D = case.q.shape
    g = torch.Generator().manual_seed(1880)
    e = torch.randint(-40, 9, (T, H, 1), generator=g).float()
    q = case.q.float() * torch.pow(2.0, e).to(DEV)
    spike = torch.rand(T, H, generator=g).to(DEV) < 0.25
    col = torch.randint(0, D, (T, H), generator=g).to(DEV)
    q[spike] = q[spike] * 1e-4
    q[spike, col[spike]] = 300.0 * torch.sign(torch.randn(int(spike.sum()), device=DEV))
    case.q.copy_(q.to(case.q.dtype))
    _check(case, _gpu(case))
