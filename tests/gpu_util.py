"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the float64 oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle
import paged_varlen_attention_attn_gb300 as pa
import workloads as W

# Tolerances of the spec (bf16 KV: max-abs, mean-abs; e4m3 KV: max-abs).
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
FP8_MAX_ABS = 6e-2


def run_gpu(case, num_splits=0, out=None, check_status=True):
    s = case.spec
    if out is None:
        out = torch.zeros_like(case.q)
    pa.forward(case.q, case.kv_cache, case.block_table, case.seq_lens, case.query_start_loc,
               scale=case.scale, num_heads=s.num_heads, num_kv_heads=s.num_kv_heads,
               head_size=s.head_size, block_size=s.block_size, window=s.window,
               causal=s.causal, kv_dtype=s.kv_dtype,
               kv_scale=case.kv_scale if s.kv_dtype else None,
               max_query_len=case.max_query_len, max_seq_len=case.max_seq_len,
               num_splits=num_splits or s.num_splits, out=out)
    if check_status:
        st = pa.pattn_read_device_status(pa.forward.last_ext)
        assert st == 0, pa.pattn_status_string(st)
    torch.cuda.synchronize()
    return out


def _host(case, kv=None, bt=None):
    q = case.q.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    kv = case.kv_cache if kv is None else kv
    kv = kv.detach().cpu()
    kv = kv.view(torch.int16).numpy().view(np.uint16) if case.spec.kv_dtype != 1 else kv.numpy()
    bt = (case.block_table if bt is None else bt).cpu().numpy()
    return q, kv, bt, case.seq_lens.cpu().numpy(), case.query_start_loc.cpu().numpy()


def oracle_kwargs(case):
    s = case.spec
    return dict(scale=case.scale, num_heads=s.num_heads, num_kv_heads=s.num_kv_heads,
                head_size=s.head_size, block_size=s.block_size, window=s.window,
                causal=s.causal, kv_dtype=s.kv_dtype, kv_scale=case.kv_scale)


def oracle_all(case):
    q, kv, bt, sl, qsl = _host(case)
    return oracle.ref_varlen(q, kv, bt, sl, qsl, **oracle_kwargs(case))


def oracle_sampled(case, rows):
    """Oracle for (token, head) rows of a large case: only the KV blocks of the
    requests those rows belong to are copied to the host (block ids remapped)."""
    qsl = case.query_start_loc.cpu().numpy()
    sl = case.seq_lens.cpu().numpy()
    bs = case.spec.block_size
    req = sorted({int(np.searchsorted(qsl, t, side="right") - 1) for t, _ in rows})
    bt_full = case.block_table.cpu()
    blocks = []
    for r in req:
        n = (int(sl[r]) + bs - 1) // bs
        blocks.extend(int(b) for b in bt_full[r, :n])
    uniq = sorted(set(blocks))
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.tensor(uniq, dtype=torch.long, device=case.kv_cache.device)
    kv_small = case.kv_cache.index_select(1, idx)
    bt_small = torch.zeros_like(bt_full)
    for r in req:
        n = (int(sl[r]) + bs - 1) // bs
        bt_small[r, :n] = torch.tensor([remap[int(b)] for b in bt_full[r, :n]], dtype=torch.int32)
    q, kv, bt, sl_, qsl_ = _host(case, kv=kv_small, bt=bt_small)
    return oracle.ref_rows(q, kv, bt, sl_, qsl_, rows=np.asarray(rows, dtype=np.int32),
                           **oracle_kwargs(case))


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), "non-finite GPU output"
    d = np.abs(got - ref)
    return float(d.max()), float(d.mean())


def assert_close(got, ref, kv_dtype):
    mx, mean = errors(got, ref)
    if kv_dtype != W.KV_FP8_E4M3:  # 16-bit caches: bf16's tolerance
        assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS, (mx, mean)
    else:
        assert mx <= FP8_MAX_ABS, (mx, mean)
    return mx, mean


def valid_rows(case):
    qsl = case.query_start_loc.cpu().numpy()
    return int(qsl[0]), int(qsl[-1])


def check_case(case, num_splits=0):
    out = run_gpu(case, num_splits=num_splits)
    ref, _ = oracle_all(case)
    a, b = valid_rows(case)
    got = out[a:b].float().cpu().numpy()
    return assert_close(got, ref[a:b], case.spec.kv_dtype)
