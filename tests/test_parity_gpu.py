"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.  Tolerances: bf16 KV max-abs 2e-2 and mean-abs 2e-3;
e4m3 KV max-abs 6e-2.  Small cases compare every row; the full-size workloads
compare sampled rows (the oracle recomputes each one from the definition)."""
import numpy as np
import pytest
import torch

import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from cases import shuffle_blocks, small_spec
from gpu_util import (assert_close, check_case, oracle_all, oracle_sampled, run_gpu,
                      valid_rows)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_varlen_attention_attn_gb300 import _build
    _build.build()
    pa.load()


def make(spec):
    return W.make_case(spec, device=DEV)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_small(G, D):
    Hkv = 2
    spec = small_spec(300 + G * 7 + D, H=G * Hkv, Hkv=Hkv, d=D, bs=16, n_req=5, max_s=300,
                      kinds=("decode",))
    check_case(make(spec))


@pytest.mark.parametrize("splits", [1, 2, 3, 16, 64])
def test_decode_forced_splits(splits):
    spec = small_spec(400 + splits, H=8, Hkv=2, d=128, bs=16, n_req=6, max_s=700,
                      kinds=("decode",))
    check_case(make(spec), num_splits=splits)


@pytest.mark.parametrize("bs", [16, 32, 64, 256])
@pytest.mark.parametrize("window", [0, 1, 7, 100])
def test_decode_block_sizes_and_windows(bs, window):
    spec = small_spec(500 + bs + window, H=8, Hkv=2, d=128, bs=bs, n_req=5, max_s=600,
                      window=window, kinds=("decode",))
    check_case(make(spec))


@pytest.mark.parametrize("splits", [1, 16])
def test_decode_fp8(splits):
    spec = small_spec(600 + splits, H=16, Hkv=2, d=128, bs=64, n_req=4, max_s=2000,
                      kv_dtype=W.KV_FP8_E4M3, kinds=("decode",))
    check_case(make(spec), num_splits=splits)


@pytest.mark.parametrize("G,D", [(8, 128), (16, 64), (4, 128)])
def test_decode_fp8_query_heads_of_very_different_magnitudes(G, D):
    # The e4m3 decode scores are 8-bit MMAs on the K codes against each head's
    # q split into e4m3 hi + lo codes after a power-of-two scaling; heads
    # scaled from 2^-40 to 2^8 (and heads with one large entry among small
    # ones) must still match the definition.
    spec = small_spec(640 + G + D, H=2 * G, Hkv=2, d=D, bs=16, n_req=6, max_s=900,
                      kv_dtype=W.KV_FP8_E4M3, kinds=("decode",))
    case = make(spec)
    T, H, _ = case.q.shape
    g = torch.Generator().manual_seed(640 + G)
    e = torch.randint(-40, 9, (T, H, 1), generator=g).float()
    q = case.q.float() * torch.pow(2.0, e).to(DEV)
    spike = torch.rand(T, H, generator=g).to(DEV) < 0.25
    col = torch.randint(0, D, (T, H), generator=g).to(DEV)
    q[spike] = q[spike] * 1e-4
    q[spike, col[spike]] = 300.0 * torch.sign(torch.randn(int(spike.sum()), device=DEV))
    case.q.copy_(q.to(case.q.dtype))
    check_case(case)


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_FP8_E4M3])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Hkv", [1, 2, 4, 8])
@pytest.mark.parametrize("G", [4, 16])
def test_decode_every_kernel_shape(G, Hkv, D, kv_dtype):
    """Every decode kernel instance: head size x KV dtype x KV heads per CTA
    (4, 2 or 1, set by Hkv and the stage size) x one or two head tiles (G up
    to 8 or above), with partitions and a ragged last page."""
    spec = small_spec(800 + G * 31 + Hkv * 7 + D + kv_dtype, H=G * Hkv, Hkv=Hkv, d=D,
                      bs=16, n_req=3, max_s=700, kv_dtype=kv_dtype, kinds=("decode",))
    check_case(make(spec), num_splits=3)


def test_decode_noncausal():
    spec = small_spec(610, H=8, Hkv=2, d=64, bs=16, n_req=4, max_s=300, causal=0,
                      kinds=("decode",))
    check_case(make(spec))


# ------------------------------------------------------------------ prefill

@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 64, 128, 256])
def test_prefill_small(D, bs):
    spec = small_spec(700 + D + bs, H=4, Hkv=2, d=D, bs=bs, n_req=3, max_s=400,
                      kinds=("prefill",))
    check_case(make(spec))


@pytest.mark.parametrize("window", [1, 5, 128, 200])
def test_prefill_window(window):
    spec = small_spec(800 + window, H=4, Hkv=1, d=128, bs=16, n_req=3, max_s=600,
                      window=window, kinds=("prefill", "chunk"))
    check_case(make(spec))


def test_prefill_noncausal():
    spec = small_spec(820, H=4, Hkv=2, d=128, bs=32, n_req=3, max_s=400, causal=0,
                      kinds=("prefill", "chunk"))
    check_case(make(spec))


@pytest.mark.parametrize("H,Hkv,D,window", [(3, 1, 128, 0), (6, 2, 64, 0), (3, 3, 128, 200),
                                             (5, 1, 128, 96), (1, 1, 64, 0)])
def test_prefill_odd_group_row_tile_pairs(H, Hkv, D, window):
    # An odd GQA ratio makes a work item two consecutive 128-row tiles of one
    # head, whose key ranges differ (the second tile's causal range reaches one
    # tile further, and under a window the first one's starts earlier): one
    # sub-tile has no MMAs for some key tiles of the item, and the two MMA
    # issuers still take turns over every tile.  Rows span several tile pairs
    # with ragged tails, and single-tile items leave the second sub-tile empty.
    spec = small_spec(1000 + 37 * H + 11 * Hkv + D + window, H=H, Hkv=Hkv, d=D, bs=16,
                      n_req=4, max_s=700, window=window, kinds=("prefill", "chunk", "decode"))
    check_case(make(spec))


@pytest.mark.parametrize("seed", range(6))
def test_mixed_batches(seed):
    spec = small_spec(900 + seed, H=8, Hkv=2, d=128, bs=16, n_req=7, max_s=520,
                      window=[0, 64][seed % 2], kinds=("prefill", "decode", "chunk", "empty"))
    check_case(make(spec))


def test_tiles_span_several_and_ragged_tail():
    # 3 x 128 + 37 query rows, chunked on 300 cached tokens
    spec = W.CaseSpec("ragged", [421, 1, 129], [721, 50, 129], 8, 2, 128, 16, seed=77)
    check_case(make(spec))


def test_tiny_mixed_workload_all_rows():
    check_case(make(W.config_spec(1)))


def test_decode_first_and_prefill_first_orders_agree():
    a = W.CaseSpec("pf_first", [64, 1, 1], [100, 300, 90], 8, 2, 128, 16, seed=88)
    case = make(a)
    out1 = run_gpu(case)
    # same requests, decodes first
    order = [1, 2, 0]
    ql = [a.q_lens[i] for i in order]
    qsl = torch.zeros(4, dtype=torch.int32)
    qsl[1:] = torch.cumsum(torch.tensor(ql), 0)
    old = case.query_start_loc.cpu()
    q2 = torch.cat([case.q[int(old[i]):int(old[i + 1])] for i in order])
    case2 = W.Case(spec=W.CaseSpec("dec_first", ql, [a.seq_lens[i] for i in order], 8, 2, 128,
                                   16, seed=88),
                   q=q2, kv_cache=case.kv_cache, block_table=case.block_table[order].contiguous(),
                   seq_lens=case.seq_lens[order].contiguous(), query_start_loc=qsl.to(DEV),
                   scale=case.scale)
    out2 = run_gpu(case2)
    back = torch.cat([out2[2:66], out2[0:1], out2[1:2]])
    assert torch.equal(out1, back)


# ------------------------------------------------------------------ invariants on the GPU

def test_block_shuffle_is_bitwise_invariant_on_gpu():
    spec = small_spec(1000, H=8, Hkv=2, d=128, bs=16, n_req=6, max_s=500, extra_pool=20,
                      kinds=("prefill", "decode", "chunk"))
    case = make(spec)
    a = run_gpu(case)
    b = run_gpu(shuffle_blocks(case, 5))
    assert torch.equal(a, b)


def test_poisoned_unused_slots_and_blocks():
    spec = small_spec(1100, H=8, Hkv=2, d=128, bs=16, n_req=6, max_s=500, extra_pool=10,
                      kinds=("prefill", "decode", "chunk"))
    case = make(spec)
    ref = run_gpu(case).clone()
    kv = case.kv_cache.clone()
    bs = spec.block_size
    used = set()
    for r in range(case.num_seqs):
        s = int(case.seq_lens[r])
        nb = (s + bs - 1) // bs
        used.update(int(b) for b in case.block_table[r, :nb])
        last = int(case.block_table[r, nb - 1])
        kv[:, last, s - (nb - 1) * bs:] = float("nan")
    for b in range(kv.shape[1]):
        if b not in used:
            kv[:, b] = float("nan")
    pc = W.Case(spec=spec, q=case.q, kv_cache=kv, block_table=case.block_table,
                seq_lens=case.seq_lens, query_start_loc=case.query_start_loc, scale=case.scale)
    got = run_gpu(pc)
    assert torch.equal(ref, got)


def test_window_at_least_seq_len_equals_full_on_gpu():
    spec = small_spec(1200, H=8, Hkv=2, d=128, bs=16, n_req=5, max_s=300,
                      kinds=("prefill", "decode", "chunk"))
    case = make(spec)
    full = run_gpu(case)
    spec_w = W.CaseSpec(**{**spec.__dict__, "window": 300})
    case_w = W.Case(spec=spec_w, q=case.q, kv_cache=case.kv_cache,
                    block_table=case.block_table, seq_lens=case.seq_lens,
                    query_start_loc=case.query_start_loc, scale=case.scale)
    assert torch.equal(full, run_gpu(case_w))


def test_split_count_changes_only_rounding():
    spec = small_spec(1300, H=8, Hkv=2, d=128, bs=16, n_req=6, max_s=3000, kinds=("decode",))
    case = make(spec)
    a = run_gpu(case, num_splits=1).float()
    b = run_gpu(case, num_splits=16).float()
    assert (a - b).abs().max().item() <= 1e-2


# ------------------------------------------------------------------ full-size workloads

def _sample_rows(case, n_per_req=3, heads=None, max_reqs=12, seed=0):
    rng = np.random.default_rng(seed)
    qsl = case.query_start_loc.cpu().numpy()
    H = case.spec.num_heads
    B = len(qsl) - 1
    reqs = sorted(set([0, B - 1] + list(rng.choice(B, size=min(B, max_reqs), replace=False))))
    rows = []
    for r in reqs:
        t0, t1 = int(qsl[r]), int(qsl[r + 1])
        if t1 == t0:
            continue
        cand = {t0, t1 - 1}
        if t1 - t0 > 1:
            for edge in (127, 128, 255, 256):
                if t0 + edge < t1:
                    cand.add(t0 + edge)
            cand.update(int(x) for x in rng.integers(t0, t1, size=n_per_req))
        hs = heads if heads is not None else sorted(set([0, H - 1] + list(rng.integers(0, H, 2))))
        for t in sorted(cand):
            for h in hs:
                rows.append((t, h))
    return rows


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_full_size_workload_sampled_rows(cfg):
    case = make(W.config_spec(cfg))
    out = run_gpu(case)
    rows = _sample_rows(case, seed=cfg)
    ref, _ = oracle_sampled(case, rows)
    t = torch.tensor([r[0] for r in rows], device=DEV)
    h = torch.tensor([r[1] for r in rows], device=DEV)
    got = out[t, h].float().cpu().numpy()
    assert_close(got, ref, case.spec.kv_dtype)
    assert torch.isfinite(out.float()).all()
    del case, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", [3, 4])
def test_full_size_workload_over_an_e4m3_cache_sampled_rows(cfg):
    # the varlen prefill and the mixed workload (co-scheduled kernels) with
    # their caches quantised to e4m3: the prefill rows take the 8-bit score
    # MMAs against the split q, the decode rows the widening decode kernel
    import dataclasses
    case = make(dataclasses.replace(W.config_spec(cfg), kv_dtype=W.KV_FP8_E4M3))
    out = run_gpu(case)
    rows = _sample_rows(case, seed=10 + cfg)
    ref, _ = oracle_sampled(case, rows)
    t = torch.tensor([r[0] for r in rows], device=DEV)
    h = torch.tensor([r[1] for r in rows], device=DEV)
    got = out[t, h].float().cpu().numpy()
    assert_close(got, ref, W.KV_FP8_E4M3)
    assert torch.isfinite(out.float()).all()
    del case, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_FP8_E4M3])
@pytest.mark.parametrize("D", [128, 64])
def test_query_row_with_a_nan_gives_nan_there_only(kv_dtype, D):
    # The definition makes a (row, head) whose q holds a NaN all NaN (every
    # score is NaN); every path must give NaN there, whatever its operand
    # handling (f16 q, the e4m3 split into hi + lo codes), and leave the other
    # rows exact.
    spec = small_spec(1400 + D + kv_dtype, H=8, Hkv=2, d=D, bs=16, n_req=6, max_s=500,
                      kv_dtype=kv_dtype)
    case = make(spec)
    T = case.q.shape[0]
    g = torch.Generator().manual_seed(1400 + D)
    bad = [(int(t), int(h)) for t, h in zip(torch.randint(0, T, (6,), generator=g),
                                            torch.randint(0, 8, (6,), generator=g))]
    qsl = case.query_start_loc.cpu().numpy()
    bad.append((int(qsl[-1]) - 1, 3))  # the last request's last row
    for t, h in bad:
        case.q[t, h, (t * 7 + h) % D] = float("nan")
    out = run_gpu(case).float().cpu().numpy()
    ref, _ = oracle_all(case)
    a, b = valid_rows(case)
    keep = np.zeros(out.shape[:2], dtype=bool)
    keep[a:b] = True
    for t, h in bad:
        if a <= t < b:
            assert np.isnan(out[t, h]).all(), (t, h)
            assert np.isnan(ref[t, h]).all(), (t, h)
        keep[t, h] = False
    assert np.isfinite(ref[keep]).all()
    assert_close(out[keep], ref[keep], kv_dtype)


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_FP8_E4M3])
def test_one_long_prefill_and_a_long_chunk_sampled_rows(kv_dtype):
    # a 32,768-token prefill (256 key tiles for its last row tiles) and a
    # 4,096-token chunk on 28,672 cached tokens beside two decodes: long items
    # that cross many ring stages, and few enough items that CTAs claim most
    # of them at run time; rows sampled at tile edges against the oracle
    q_lens = [32768, 4096, 1, 1]
    seq = [32768, 32768, 32768, 9000]
    spec = W.CaseSpec("long_prefill", q_lens, seq, 8, 2, 128, 16, kv_dtype=kv_dtype,
                      pool_blocks=sum((s + 15) // 16 for s in seq) + 8, seed=1500 + kv_dtype)
    case = make(spec)
    out = run_gpu(case)
    rows = _sample_rows(case, n_per_req=4, seed=1500)
    qsl = case.query_start_loc.cpu().numpy()
    rows += [(int(qsl[0]) + 32767, 5), (int(qsl[1]) + 4095, 2)]  # the longest rows
    ref, _ = oracle_sampled(case, rows)
    t = torch.tensor([r[0] for r in rows], device=DEV)
    h = torch.tensor([r[1] for r in rows], device=DEV)
    assert_close(out[t, h].float().cpu().numpy(), ref, kv_dtype)
    assert torch.isfinite(out.float()).all()
    del case, out
    torch.cuda.empty_cache()
