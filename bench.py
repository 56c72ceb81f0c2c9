#!/usr/bin/env python3
"""Benchmark of the paged varlen attention library on one or more GB300s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

One step = one pattn_varlen_fwd call (plan, prefill, decode, combine -- every
phase the workload needs) over one synthetic batch already resident in HBM.
The default workload is the largest one, the mixed batch that exercises both
kernels: 4 chunked prefills of 2048 new tokens on 6144 cached ones plus 192
decodes with seq_len ~ U{1024..32768}, sliding window 4096, 64 query / 8 KV
heads, head 128, block 16 (13.4 GB cache).  --config 1..5 selects the other
workloads.  Prints ONE JSON line.

value: the step's fraction of its roofline, in percent: the roofline time
max(F / P_tensor, B / BW_hbm) of the step's algorithmic work (F: unmasked
prefill FLOPs, 4 d per visible (row, key, head); B: visible decode K/V bytes,
the prefill requests' visible K/V bytes, q and out) divided by the measured
step time.  The line also carries each kernel's own roofline (prefill TFLOP/s
against the bf16 tensor peak, decode KV GB/s against HBM) from its own
event-timed duration.

Timing: W warm-up steps, then K steps, each bracketed by CUDA events on the
library's stream; L2 is flushed before every step, outside the events: a
256 MiB write, then a 256 MiB read of another buffer, so each step starts with
a cold L2 that holds no dirty lines (whose write-back the step would
otherwise pay for).  The timed steps carry no events between their kernels.
The dominant kernel's own duration comes from a second pass of K steps with
the library's per-phase events (pattn_ext_t.timing_events) recorded on the
same stream; with events between them the kernels run one after another.
Under torchrun (N > 1) every rank runs the same workload on its own GPU (the
path has no exchange step: replicas, weak scaling); time is the max over ranks.

--impl reference times the float64 CPU oracle (oracle/) on the host cores on a
bounded sample of the same workload, with the same metric and unit.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged attn: prefill TFLOP/s & decode KV GB/s, % of GB300 roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = {
    "decode": ["paged_varlen_attention_attn_gb300/csrc/decode.cu",
               "paged_varlen_attention_attn_gb300/csrc/common.cuh"],
    "prefill": ["paged_varlen_attention_attn_gb300/csrc/prefill.cu",
                "paged_varlen_attention_attn_gb300/csrc/common.cuh"],
    "diffkv": ["paged_varlen_attention_attn_gb300/csrc/diffkv_decode.cu",
               "paged_varlen_attention_attn_gb300/csrc/common.cuh"],
}


# ---------------------------------------------------------------- work counts

def visible_per_row(spec):
    """Keys each query row may attend to (host copy of the lengths only)."""
    dec, pre = [], []
    for ql, s in zip(spec.q_lens, spec.seq_lens):
        if ql <= 0:
            continue
        p = (s - ql) + np.arange(ql, dtype=np.int64)
        hi = np.minimum(p + 1, s) if spec.causal else np.full(ql, s, dtype=np.int64)
        lo = np.maximum(0, p - spec.window + 1) if spec.window > 0 else np.zeros(ql, np.int64)
        v = np.maximum(0, hi - lo)
        (dec if ql == 1 else pre).append(v)
    cat = lambda xs: np.concatenate(xs) if xs else np.zeros(0, np.int64)
    return cat(dec), cat(pre)


def work_counts(spec):
    """Algorithmic work of one step: prefill FLOPs (unmasked only, 4*d per key
    and head), decode KV bytes (visible tokens only), query tokens."""
    es = 1 if spec.kv_dtype == 1 else 2
    dec, pre = visible_per_row(spec)
    flops_prefill = 4.0 * spec.head_size * spec.num_heads * float(pre.sum())
    flops_decode = 4.0 * spec.head_size * spec.num_heads * float(dec.sum())
    bytes_decode = float(dec.sum()) * 2 * spec.num_kv_heads * spec.head_size * es
    # prefill K/V bytes: each request's visible key range read once
    bytes_prefill = 0.0
    for ql, s in zip(spec.q_lens, spec.seq_lens):
        if ql > 1:
            lo = max(0, s - ql - spec.window + 1) if spec.window > 0 else 0
            bytes_prefill += (s - lo) * 2 * spec.num_kv_heads * spec.head_size * es
    tokens = int(sum(spec.q_lens))
    qo_bytes = 2.0 * tokens * spec.num_heads * spec.head_size * 2
    return dict(flops_prefill=flops_prefill, flops_decode=flops_decode,
                bytes_decode=bytes_decode, bytes_prefill=bytes_prefill, bytes_qo=qo_bytes,
                tokens=tokens, row_keys=float(spec.num_heads) * float(dec.sum() + pre.sum()),
                decode_rows=int(len(dec)), prefill_rows=int(len(pre)))


def roofline_seconds(counts, pk):
    """The step's roofline time: max(F / P_tensor, B / BW) over its algorithmic
    work (prefill FLOPs; every visible K/V byte, q and out)."""
    f = counts["flops_prefill"] / (pk["bf16_tflops"] * 1e12)
    b = (counts["bytes_decode"] + counts["bytes_prefill"] + counts["bytes_qo"]) / (pk["hbm_gbs"] * 1e9)
    return max(f, b)


def has_prefill_rows(spec):
    return any(q > 1 for q in spec.q_lens)


def peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash(kind):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kind, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(PROFILE_DIR, f"{kind}_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("source_sha256_16") != kernel_hash(kind):
        return None
    try:
        return float(fields["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- distributed

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(backend):
    import torch.distributed as dist
    ws, rank, _ = dist_info()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x, device="cpu"):
    """Max of a float over ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, device="cpu"):
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(units_local, seconds_local, device="cpu"):
    """Whole-job throughput: units of all ranks / slowest rank's time."""
    total = sum_over_ranks(units_local, device)
    slowest = max_over_ranks(seconds_local, device)
    return total / slowest if slowest > 0 else 0.0, slowest


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed loop runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def call_args(case):
    s = case.spec
    return dict(scale=case.scale, num_heads=s.num_heads, num_kv_heads=s.num_kv_heads,
                head_size=s.head_size, block_size=s.block_size, window=s.window,
                causal=s.causal, kv_dtype=s.kv_dtype,
                kv_scale=case.kv_scale if s.kv_dtype == 1 else None,
                max_query_len=case.max_query_len, max_seq_len=case.max_seq_len,
                num_splits=s.num_splits)


def run_ours(args, spec, world, rank, local_rank):
    import torch
    import paged_varlen_attention_attn_gb300 as pa
    import workloads as W

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    pa.load()
    case = W.make_case(spec, device=dev)
    counts = work_counts(spec)
    stream = torch.cuda.Stream(dev)
    out = torch.empty_like(case.q)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another: cold and clean
        flush_w.zero_()
        flush_r.sum()
    ca = call_args(case)
    ws = pa.Workspace()

    def step(events=None):
        pa.forward(case.q, case.kv_cache, case.block_table, case.seq_lens,
                   case.query_start_loc, out=out, stream=stream, workspace=ws,
                   timing_events=events, **ca)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2()
            step()
    torch.cuda.synchronize()
    st = pa.pattn_read_device_status(pa.forward.last_ext)
    if st != 0:
        raise RuntimeError("device status after warm-up: " + pa.pattn_status_string(st))
    splits = pa.pattn_decode_splits(pa.forward.last_ext, spec.num_heads, spec.num_kv_heads,
                                    spec.block_size, spec.window)
    # the prefill grid the plan kernel kept for the co-scheduled step (the
    # workspace header's third word; 0 = every SM)
    prefill_ctas = int(ws.buf[8:12].view(torch.int32).item()) if has_prefill_rows(spec) else 0

    K = args.steps
    t_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(K)]
    p_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(K)]
    with torch.cuda.stream(stream):   # materialise the raw event handles
        for pe in p_ev:
            for e in pe:
                e.record()
    torch.cuda.synchronize()
    # Only the phases that are reported get events (an event pair between
    # kernels costs ~2 us of the step): the prefill and/or decode kernels.
    has_prefill = case.max_query_len > 1
    has_decode = any(q == 1 for q in spec.q_lens)
    timed = {"prefill": has_prefill, "decode": has_decode}
    handles = [[e.cuda_event if timed.get(pa.PHASES[k // 2], False) else 0
                for k, e in enumerate(pe)] for pe in p_ev]

    clocks = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    wall0 = time.perf_counter()
    # The steps are timed as a user runs them: no events between the kernels
    # (the decode kernel overlaps the kernel before it).
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_l2()
            t_ev[i][0].record()
            step()
            t_ev[i][1].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    # Kernel durations for the roofline: a second pass of the same steps with
    # events around the reported kernels (which then run one after another).
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_l2()
            step(handles[i])
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()

    step_ms = [a.elapsed_time(b) for a, b in t_ev]
    phase_ms = {name: ([pe[2 * k].elapsed_time(pe[2 * k + 1]) for pe in p_ev]
                       if timed.get(name, False) else [0.0])
                for k, name in enumerate(pa.PHASES) if name in timed}
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, device=dev)
    # plan + prefill when there are prefill rows (else the kernel that clears
    # the status word and the partition counters), decode (which also merges
    # the partitions)
    launches_per_step = (2 if has_prefill else 1) + 1

    # e2e: all inputs from pinned host memory, result read back, every step
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, case, spec, counts, dev, stream, ca, ws)

    return dict(case=case, counts=counts, ms=ms_max, ms_local=ms, ms_min=min(step_ms),
                ms_median=statistics.median(step_ms), prefill_ctas=prefill_ctas,
                wall=wall, phase_ms={k: statistics.mean(v) for k, v in phase_ms.items()},
                clocks=clk, splits=splits, launches=launches_per_step * K, e2e=e2e)


def run_e2e(args, case, spec, counts, dev, stream, ca, ws):
    """A serving loop through the public API, from host memory: the KV pool
    stays resident on the GPU (it is the cache earlier steps filled); every
    step copies from pinned host memory (one packed buffer, one copy) the
    queries, the new tokens' key and value rows and their slots, and the
    metadata, writes the new rows into the cache (pattn_reshape_and_cache),
    runs attention (pattn_varlen_fwd) and reads the output back.  The new
    tokens are each request's query positions ctx .. s-1, so the cache write
    touches exactly the slots the step's queries own.  Consecutive steps use
    two buffer slots so that one step's copies overlap its neighbours'
    compute; the time per step is the span of K steps over K."""
    import torch
    import paged_varlen_attention_attn_gb300 as pa
    bt = case.block_table.cpu()
    bs = spec.block_size
    slots = []
    for r, (q, s) in enumerate(zip(spec.q_lens, spec.seq_lens)):
        k = torch.arange(s - q, s)
        slots.append(bt[r, k // bs].to(torch.int64) * bs + k % bs)
    slots = torch.cat(slots)
    T, Hkv, d = int(slots.numel()), spec.num_kv_heads, spec.head_size
    g = torch.Generator().manual_seed(spec.seed + 11)
    kv_dt = torch.float16 if spec.kv_dtype == 2 else torch.bfloat16
    new_k = torch.randn(T, Hkv, d, generator=g).to(kv_dt)
    new_v = torch.randn(T, Hkv, d, generator=g).to(kv_dt)
    parts = {"q": case.q.cpu(), "new_k": new_k, "new_v": new_v, "slots": slots,
             "block_table": case.block_table.cpu(), "seq_lens": case.seq_lens.cpu(),
             "query_start_loc": case.query_start_loc.cpu()}
    # The inputs of a step travel in one pinned buffer and one copy, as a
    # serving engine packs them, each part at a 256-byte aligned offset; the
    # device side holds views into one device buffer.
    offs, total = {}, 0
    for k, v in parts.items():
        offs[k] = total
        total += (v.numel() * v.element_size() + 255) // 256 * 256
    host_all = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_all = torch.empty(total, dtype=torch.uint8, device=dev)
    dev_bufs = {}
    for k, v in parts.items():
        n = v.numel() * v.element_size()
        host_all[offs[k]:offs[k] + n].copy_(v.contiguous().view(-1).view(torch.uint8))
        dev_bufs[k] = dev_all[offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
    h2d = sum(v.numel() * v.element_size() for v in parts.values())
    d2h = case.q.numel() * case.q.element_size()
    ks = case.kv_scale if spec.kv_dtype == 1 else None
    K = max(3, min(args.steps, args.e2e_steps))
    # Two slots, as a serving loop runs: step i's inputs go up (h2d stream)
    # while step i-1 computes; its output comes back (d2h stream) while step
    # i+1 computes.  A slot's buffers are reused only after the work that
    # used them two steps earlier is done (events).  Every step still copies
    # all of its own inputs and reads back its output inside the timed region.
    dev_alls = [dev_all, torch.empty_like(dev_all)]
    views = []
    for da in dev_alls:
        v = {}
        for k, t in parts.items():
            n = t.numel() * t.element_size()
            v[k] = da[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
        views.append(v)
    outs = [torch.empty_like(case.q) for _ in range(2)]
    out_hosts = [torch.empty(case.q.shape, dtype=case.q.dtype).pin_memory() for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    up_done = [ev() for _ in range(K + 2)]
    comp_done = [ev() for _ in range(K + 2)]
    down_done = [ev() for _ in range(K + 2)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def run(n, timed):
        if timed:
            t0.record(s_h2d)
        for i in range(n):
            sl = i % 2
            with torch.cuda.stream(s_h2d):
                if i >= 2:
                    s_h2d.wait_event(comp_done[i - 2])   # slot's inputs no longer read
                dev_alls[sl].copy_(host_all, non_blocking=True)
                up_done[i].record(s_h2d)
            with torch.cuda.stream(stream):
                stream.wait_event(up_done[i])
                if i >= 2:
                    stream.wait_event(down_done[i - 2])  # slot's output read back
                v = views[sl]
                pa.reshape_and_cache(v["new_k"], v["new_v"], case.kv_cache, v["slots"],
                                     block_size=bs, kv_dtype=spec.kv_dtype, kv_scale=ks,
                                     stream=stream)
                pa.forward(v["q"], case.kv_cache, v["block_table"], v["seq_lens"],
                           v["query_start_loc"], out=outs[sl], stream=stream, workspace=ws, **ca)
                comp_done[i].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(comp_done[i])
                out_hosts[sl].copy_(outs[sl], non_blocking=True)
                down_done[i].record(s_d2h)
        if timed:
            s_h2d.wait_stream(s_d2h)
            s_h2d.wait_stream(stream)
            t1.record(s_h2d)

    run(2, False)
    torch.cuda.synchronize()
    run(K, True)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / K
    ms = max_over_ranks(ms, device=dev)
    del dev_bufs, dev_all, dev_alls, host_all
    return dict(ms=ms, h2d=h2d, d2h=d2h, pipelined=True)


# ---------------------------------------------------------------- oracle (CPU)

def oracle_sample(case, spec, stride):
    """Host arrays and (token, head) rows of a bounded, uniform sample of the
    workload: every stride-th decode request and, of each prefill request,
    every stride-th query row (all heads of each chosen token).  Only the KV
    blocks the chosen rows can see are copied to the host (block ids remapped;
    the oracle reads no other block)."""
    import torch
    qsl = case.query_start_loc.cpu().numpy()
    sl = case.seq_lens.cpu().numpy()
    H, bs, W = spec.num_heads, spec.block_size, spec.window
    toks, need, n_dec = [], {}, 0
    for r in range(len(sl)):
        t0, ql, s = int(qsl[r]), int(qsl[r + 1] - qsl[r]), int(sl[r])
        if ql <= 0:
            continue
        if ql == 1:
            pick = [0] if n_dec % stride == 0 else []
            n_dec += 1
        else:
            pick = list(range(stride // 2 if ql > stride // 2 else 0, ql, stride))
        if not pick:
            continue
        ctx = s - ql
        lo = min(max(0, ctx + i - W + 1) if W > 0 else 0 for i in pick)
        hi = max(min(s, ctx + i + 1) if spec.causal else s for i in pick)
        need[r] = (lo // bs, (hi + bs - 1) // bs)
        toks.extend(t0 + i for i in pick)
    bt_full = case.block_table.cpu()
    blocks = sorted({int(b) for r, (a, e) in need.items() for b in bt_full[r, a:e]})
    remap = {b: i for i, b in enumerate(blocks)}
    kv = case.kv_cache.index_select(1, torch.tensor(blocks, device=case.kv_cache.device)).cpu()
    bt = torch.zeros_like(bt_full)
    for r, (a, e) in need.items():
        bt[r, a:e] = torch.tensor([remap[int(b)] for b in bt_full[r, a:e]], dtype=torch.int32)
    q = case.q.cpu().view(torch.int16).numpy().view(np.uint16)
    kvn = kv.view(torch.int16).numpy().view(np.uint16) if spec.kv_dtype != 1 else kv.numpy()
    rows = np.array([(t, h) for t in toks for h in range(H)], np.int32).reshape(-1, 2)
    return dict(q=q, kv=kvn, bt=bt.numpy(), sl=sl, qsl=qsl, rows=rows, tokens=len(toks))


def sample_row_keys(spec, qsl, rows):
    """Visible (row, key) pairs of the sampled rows: the oracle's work."""
    qsl = np.asarray(qsl)
    r = np.searchsorted(qsl, rows[:, 0], side="right") - 1
    s = np.asarray(spec.seq_lens)[r]
    ql = np.asarray(spec.q_lens)[r]
    p = (s - ql) + (rows[:, 0] - qsl[r])
    hi = np.minimum(p + 1, s) if spec.causal else s
    lo = np.maximum(0, p - spec.window + 1) if spec.window > 0 else 0
    return float(np.maximum(0, hi - lo).sum())


def time_oracle(case, spec, stride, threads=None):
    """Wall time of the float64 oracle on a uniform 1/stride sample."""
    import oracle
    smp = oracle_sample(case, spec, stride)
    kw = dict(scale=case.scale, num_heads=spec.num_heads, num_kv_heads=spec.num_kv_heads,
              head_size=spec.head_size, block_size=spec.block_size, window=spec.window,
              causal=spec.causal, kv_dtype=spec.kv_dtype, kv_scale=case.kv_scale)
    cores = threads or os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.ref_rows(smp["q"], smp["kv"], smp["bt"], smp["sl"], smp["qsl"],
                    rows=smp["rows"], num_threads=cores, **kw)
    sec = time.perf_counter() - t0
    rk = sample_row_keys(spec, smp["qsl"], smp["rows"])
    return dict(seconds=sec, row_keys=rk, cores=cores, tokens=smp["tokens"],
                sample=f"one in {stride} decode requests and one in {stride} query rows of "
                       f"each prefill request: {smp['tokens']} of {sum(spec.q_lens)} query "
                       f"tokens x {spec.num_heads} heads, all their visible keys "
                       f"({rk:.3g} (row, key) pairs)")


def cpu_model():
    """The host CPU's model name (lscpu), for the CPU baseline."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_stride(case, spec, budget_s, threads=None):
    """The sample stride whose oracle run takes about budget_s: calibrated on
    a small sample first."""
    full = work_counts(spec)["row_keys"]
    cal_stride = max(1, int(full / 2e6))  # ~2M (row, key) pairs
    cal = time_oracle(case, spec, cal_stride, threads)
    rate = cal["row_keys"] / max(cal["seconds"], 1e-6)
    want = max(1.0, rate * budget_s)
    return max(1, int(math.ceil(full / want)))


# ---------------------------------------------------------------- metric

UNIT = "% of roofline"


def metric_value(counts, seconds, pk):
    """The metric: the step's roofline time over its measured time, percent."""
    return 100.0 * roofline_seconds(counts, pk) / seconds


def config_dict(spec, cfg, world):
    """The `config` of both arms' lines (identical, so the two are comparable)."""
    return {"workload": workload_desc(spec, cfg), "config_index": cfg,
            "l2": "flushed before every timed step (256 MiB write, then 256 MiB read)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def workload_desc(spec, cfg):
    kinds = {1: "tiny mixed batch", 2: "decode-only GQA batch", 3: "varlen causal prefill",
             4: "mixed chunked prefill + decode, sliding window 4096",
             5: "long-context split-KV decode, e4m3 KV"}
    return (f"{kinds.get(cfg, spec.name)}: {len(spec.q_lens)} requests, "
            f"query_len {min(spec.q_lens)}..{max(spec.q_lens)}, "
            f"seq_len {min(spec.seq_lens)}..{max(spec.seq_lens)}, "
            f"H {spec.num_heads}, Hkv {spec.num_kv_heads}, d {spec.head_size}, "
            f"block {spec.block_size}, window {spec.window}, "
            f"kv {['bf16', 'e4m3', 'f16'][spec.kv_dtype]}")


# ---------------------------------------------------------------- main

def run_cascade(args, world, rank, local, prefix):
    """Time pattn_cascade_fwd against pattn_varlen_fwd on a decode batch whose
    requests share a long cached prefix: 64 requests, `prefix` keys shared
    (default 32768: 134 MB of K/V, more than L2), own suffixes U{128..1024},
    H 32 / Hkv 8, d 128, block 16 (seed 1501); bf16, or f16 / e4m3 with
    --f16 / --fp8.
    value = the plain call's algorithmic KV bytes / the cascade call's time
    (effective GB/s); the line also gives both times."""
    import torch
    import paged_varlen_attention_attn_gb300 as pa
    import workloads as W
    pa.load()
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)
    B = 64
    suffix = W._uniform_ints(128, 1024, B, 1501)
    seq = [prefix + x for x in suffix]
    kv = W.KV_FP8_E4M3 if args.fp8 else (W.KV_F16 if args.f16 else W.KV_BF16)
    spec = W.CaseSpec("cascade_decode", [1] * B, seq, 32, 8, 128, 16,
                      pool_blocks=sum((s + 15) // 16 for s in seq) + 8, seed=1501, kv_dtype=kv)
    case = W.make_case(spec, device=dev)
    case.block_table[:, :prefix // 16] = case.block_table[0, :prefix // 16].clone()
    counts = work_counts(spec)
    stream = torch.cuda.Stream(dev)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = torch.empty_like(case.q)
    ws = pa.Workspace()
    kw = dict(scale=case.scale, num_heads=32, num_kv_heads=8, head_size=128, block_size=16,
              kv_dtype=kv, kv_scale=case.kv_scale if kv == W.KV_FP8_E4M3 else None,
              max_query_len=1, max_seq_len=max(seq), out=out, workspace=ws, stream=stream)

    def plain():
        pa.forward(case.q, case.kv_cache, case.block_table, case.seq_lens,
                   case.query_start_loc, **kw)

    def casc():
        pa.cascade_forward(case.q, case.kv_cache, case.block_table, case.seq_lens,
                           case.query_start_loc, common_prefix_len=prefix, **kw)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush_w.zero_(); flush_r.sum(); fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for a, b in ev:
                flush_w.zero_(); flush_r.sum()
                a.record(); fn(); b.record()
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    ms_plain = timed(plain)
    ms_casc = timed(casc)
    clk = clocks.stop()
    ms_casc = max_over_ranks(ms_casc, device=dev)
    pk, pk_src = peaks()
    gbs = counts["bytes_decode"] / (ms_casc / 1e3) / 1e9
    value, _ = aggregate(gbs * (ms_casc / 1e3), ms_casc / 1e3, device=dev)
    line = {"metric": "cascade decode: plain algorithmic KV GB/s per cascade-call time",
            "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_casc, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {0: "bf16 (fp32 accumulate)", 1: "e4m3 KV, bf16 Q/out, fp32 accumulate",
                      2: "f16 (fp32 accumulate)"}[kv], "data": "synthetic (seeded N(0,1))",
            "config": {"workload": f"{B} decode requests sharing a {prefix}-key prefix, "
                                   f"suffixes 128..1024, H 32, Hkv 8, d 128, block 16, "
                                   f"kv {['bf16', 'e4m3', 'f16'][kv]}",
                       "l2": "flushed before every timed step (256 MiB write, then 256 MiB read)"},
            "plain_ms_per_step": round(ms_plain, 5),
            "speedup_over_plain": round(ms_plain / ms_casc, 3),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                         "kernel": "whole cascade call (effective)", "peak_source": pk_src,
                         "traffic": None},
            "gpu_launches": 6 * args.steps, "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_diffkv(args, spec, world, rank, local):
    """Time pattn_varlen_fwd over a DiffKV cache (head_size_v != head_size):
    the workload's request lengths, heads and blocks, K head size 192 and V
    head size 128 in the layout [num_blocks, block_size, Hkv, 192 + 128].
    Decode batches report KV GB/s (visible keys x Hkv x (192 + 128) x 2
    bytes) against HBM; the kernel is the generic SIMT one."""
    import dataclasses
    import torch
    import paged_varlen_attention_attn_gb300 as pa
    import workloads as W
    pa.load()
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)
    dk, dv = 192, 128
    case = W.make_case(dataclasses.replace(spec, head_size=dk), device=dev)
    nb = case.kv_cache.shape[1]
    g = torch.Generator(device=dev).manual_seed(spec.seed + 11)
    cache = torch.randn(nb, spec.block_size, spec.num_kv_heads, dk + dv, generator=g,
                        device=dev).to(torch.bfloat16)
    del case.kv_cache
    vis = 0
    for q, s in zip(spec.q_lens, spec.seq_lens):
        for i in range(q):
            p = s - q + i
            lo = max(0, p - spec.window + 1) if spec.window > 0 else 0
            vis += p + 1 - lo
    nbytes = vis * spec.num_kv_heads * (dk + dv) * 2
    out = torch.empty(case.q.shape[0], spec.num_heads, dv, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    ws = pa.Workspace()

    def step():
        pa.forward(case.q, cache, case.block_table, case.seq_lens, case.query_start_loc,
                   scale=case.scale, num_heads=spec.num_heads, num_kv_heads=spec.num_kv_heads,
                   head_size=dk, block_size=spec.block_size, window=spec.window,
                   causal=spec.causal, max_query_len=case.max_query_len,
                   max_seq_len=case.max_seq_len, out=out, workspace=ws, stream=stream,
                   head_size_v=dv)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_w.zero_(); flush_r.sum(); step()
    torch.cuda.synchronize()
    st = pa.pattn_read_device_status(pa.forward.last_ext)
    if st != 0:
        raise RuntimeError("device status: " + pa.pattn_status_string(st))
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_w.zero_(); flush_r.sum()
            ev[i][0].record()
            step()
            ev[i][1].record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms = max_over_ranks(ms, device=dev)
    pk, pk_src = peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    value, _ = aggregate(gbs * (ms / 1e3), ms / 1e3, device=dev)
    line = {"metric": "DiffKV attention, KV GB/s", "value": round(value, 1),
            "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)",
            "data": "synthetic (seeded N(0,1), the workload's block tables)",
            "config": {"workload": f"{spec.name} lengths and heads, K head {dk}, V head {dv}, "
                                   f"DiffKV layout, block {spec.block_size}",
                       "l2": "flushed before every timed step (256 MiB write, then 256 MiB read)"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                         "kernel": "diffkv_decode_kernel", "peak_source": pk_src,
                         "traffic": profiled_traffic("diffkv", spec.name)},
            "gpu_launches": K, "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_cache_write(args, spec, world, rank, local):
    """Time pattn_reshape_and_cache on the workload's new tokens: request r's
    query tokens (positions ctx .. s-1) are written through its block table,
    key and value bf16 [T, Hkv, d] in, the cache's dtype out.  Algorithmic
    bytes per call: T * Hkv * d * 2 * (2 bytes read + element size written)."""
    import torch
    import paged_varlen_attention_attn_gb300 as pa
    import workloads as W
    pa.load()
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)
    case = W.make_case(spec, device=dev)
    bt = case.block_table.cpu()
    slots = []
    for r, (q, s) in enumerate(zip(spec.q_lens, spec.seq_lens)):
        k = torch.arange(s - q, s)
        slots.append(bt[r, k // spec.block_size].to(torch.int64) * spec.block_size
                     + k % spec.block_size)
    slots = torch.cat(slots).to(dev)
    T, Hkv, d = int(slots.numel()), spec.num_kv_heads, spec.head_size
    g = torch.Generator(device=dev).manual_seed(spec.seed + 7)
    key = torch.randn(T, Hkv, d, generator=g, device=dev).to(torch.bfloat16)
    value = torch.randn(T, Hkv, d, generator=g, device=dev).to(torch.bfloat16)
    es = 1 if spec.kv_dtype == 1 else 2
    nbytes = T * Hkv * d * 2 * (2 + es)
    stream = torch.cuda.Stream(dev)
    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    ks = case.kv_scale if spec.kv_dtype == 1 else None

    def step():
        pa.reshape_and_cache(key, value, case.kv_cache, slots, block_size=spec.block_size,
                             kv_dtype=spec.kv_dtype, kv_scale=ks, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_w.zero_(); flush_r.sum(); step()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_w.zero_(); flush_r.sum()
            ev[i][0].record()
            step()
            ev[i][1].record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms = max_over_ranks(ms, device=dev)
    pk, pk_src = peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    value, _ = aggregate(gbs * (ms / 1e3), ms / 1e3, device=dev)
    line = {"metric": "kv-cache write (reshape_and_cache) GB/s", "value": round(value, 1),
            "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": ("f16 in, f16" if spec.kv_dtype == 2 else "bf16 in, " + ("e4m3" if spec.kv_dtype else "bf16")) + " cache",
            "data": "synthetic (seeded N(0,1) rows, the workload's block tables)",
            "config": {"workload": f"{T} new tokens of the {spec.name} workload, Hkv {Hkv}, "
                                   f"d {d}, block {spec.block_size}",
                       "l2": "flushed before every timed step (256 MiB write, then 256 MiB read)"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                         "kernel": "reshape_and_cache_kernel", "peak_source": pk_src,
                         "traffic": None},
            "gpu_launches": K, "clocks": clk}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="CPU baseline: oracle seconds on the host cores (1-thread: a quarter)")
    ap.add_argument("--cascade-prefix", type=int, default=32768,
                    help="--op cascade: shared prefix length in keys (multiple of 16)")
    ap.add_argument("--f16", action="store_true",
                    help="run the workload with f16 q, cache and output (16-bit workloads only)")
    ap.add_argument("--fp8", action="store_true",
                    help="run the workload over an e4m3 cache (per-tensor scales)")
    ap.add_argument("--splits", type=int, default=None,
                    help="force the decode partition count (default: the workload's own, "
                         "0 = the library's choice)")
    ap.add_argument("--op", choices=["attention", "cache_write", "cascade", "diffkv"],
                    default="attention",
                    help="cache_write: time pattn_reshape_and_cache on the workload's new "
                         "tokens instead of the attention step; diffkv: the attention step "
                         "over a DiffKV cache (K head 192, V head 128)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = {1: 2000, 2: 2000, 3: 50, 4: 100, 5: 400}.get(args.config, 100)
    if args.warmup < 3:
        args.warmup = 3

    import dataclasses
    import workloads as W
    spec = W.config_spec(args.config)
    if args.f16:
        if spec.kv_dtype != W.KV_BF16:
            raise SystemExit("--f16 needs a 16-bit workload")
        spec = dataclasses.replace(spec, kv_dtype=W.KV_F16, name=spec.name + "_f16")
    if args.fp8:
        if spec.kv_dtype != W.KV_BF16:
            raise SystemExit("--fp8 needs a bf16 workload")
        spec = dataclasses.replace(spec, kv_dtype=W.KV_FP8_E4M3, name=spec.name + "_fp8")
    if args.splits is not None:
        spec = dataclasses.replace(spec, num_splits=args.splits)
    world, rank, local = dist_info()

    if args.impl == "reference":
        return run_reference(args, spec, world, rank)

    import torch
    dist_init("nccl")
    if args.op == "cache_write":
        return run_cache_write(args, spec, world, rank, local)
    if args.op == "cascade":
        return run_cascade(args, world, rank, local, args.cascade_prefix)
    if args.op == "diffkv":
        return run_diffkv(args, spec, world, rank, local)
    res = run_ours(args, spec, world, rank, local)
    line = attention_line(args, spec, world, rank, local, res)
    if rank == 0:
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_initialized():
        dist.destroy_process_group()


def kernel_roofline(kind, counts, ms, pk, pk_src, spec):
    """One kernel's roofline object from its event-timed duration."""
    if kind == "prefill":
        achieved = counts["flops_prefill"] / (ms / 1e3) / 1e12
        peak = pk["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "kernel": "prefill_kernel" + ((" (e4m3: 8-bit score MMAs on the K codes, V "
                                               "widened to f16)" if spec.head_size == 128 else
                                               " (e4m3 tiles widened to f16)")
                                              if spec.kv_dtype == 1 else ""),
                "work_per_launch": f"{counts['flops_prefill']:.6g} FLOP (4 d per visible "
                                   f"(row, key, head))"}
    else:
        achieved = counts["bytes_decode"] / (ms / 1e3) / 1e9
        peak = pk["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "kernel": "decode_split_kernel",
                "work_per_launch": f"{counts['bytes_decode']:.6g} B (2 d es per visible "
                                   f"(key, KV head))"}
    roof["kernel_ms"] = round(ms, 4)
    roof["peak_source"] = (f"{pk_src} (MEASURED_PEAKS.json)" if pk_src == "measured"
                           else pk_src)
    roof["traffic"] = profiled_traffic(kind, spec.name)
    return roof


def attention_line(args, spec, world, rank, local, res):
    pk, pk_src = peaks()
    counts = res["counts"]
    sec = res["ms"] / 1e3
    value_local = metric_value(counts, sec, pk)
    # whole job: every replica processes the same work; value = the fraction
    # of the aggregate roofline, i.e. total work / slowest replica's time
    value, _ = aggregate(value_local * sec, sec, device=f"cuda:{local}")
    ph = res["phase_ms"]
    rooflines = {k: kernel_roofline(k, counts, ph[k], pk, pk_src, spec)
                 for k in ("prefill", "decode") if ph.get(k, 0.0) > 0}
    # dominant kernel: the longer of the two
    dom = max(rooflines, key=lambda k: ph[k])
    t_roof = roofline_seconds(counts, pk)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms"], 4),
        "ms_per_step_median": round(res["ms_median"], 4),
        "ms_per_step_min": round(res["ms_min"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype":
        {0: "bf16 (fp32 accumulate)", 1: "e4m3 KV, bf16 Q/out, fp32 accumulate",
         2: "f16 (fp32 accumulate)"}[spec.kv_dtype],
        "data": "synthetic (seeded N(0,1), seeded block permutation)",
        "config": config_dict(spec, args.config, world),
        "value_definition": "100 x roofline time / step time; roofline time = "
                            "max(prefill FLOPs / bf16 tensor peak, (decode K/V + prefill K/V "
                            "+ q + out bytes) / HBM peak)",
        "step": {"roofline_ms": round(t_roof * 1e3, 4),
                 "prefill_tflop": round(counts["flops_prefill"] / 1e12, 4),
                 "hbm_gb": round((counts["bytes_decode"] + counts["bytes_prefill"]
                                  + counts["bytes_qo"]) / 1e9, 4),
                 "tokens_per_s": round(counts["tokens"] / sec, 1),
                 "prefill_tflops_over_step": round(counts["flops_prefill"] / sec / 1e12, 2),
                 "decode_gbs_over_step": round(counts["bytes_decode"] / sec / 1e9, 1)},
        "roofline": rooflines[dom],
        "rooflines": rooflines,
        "phase_ms": {k: round(v, 4) for k, v in ph.items()},
        "decode_splits": res["splits"],
        "prefill_ctas": res["prefill_ctas"],
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
    }
    if ph.get("prefill", 0.0) > 0 and ph.get("decode", 0.0) > 0:
        # the two kernels timed apart (each on every SM) against the step,
        # where they run at the same time on different SMs
        line["co_schedule"] = {
            "serial_ms": round(ph["prefill"] + ph["decode"], 4),
            "step_ms": round(res["ms"], 4),
            "overlap_ms": round(ph["prefill"] + ph["decode"] - res["ms"], 4)}
    if args.config == 1:
        line["latency_us"] = {"mean": round(res["ms"] * 1e3, 2),
                              "median": round(res["ms_median"] * 1e3, 2),
                              "min": round(res["ms_min"] * 1e3, 2)}
    if res["e2e"] is not None:
        e = res["e2e"]
        line["e2e"] = {"value": round(metric_value(counts, e["ms"] / 1e3, pk), 3),
                       "unit": UNIT,
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "ms_per_step": round(e["ms"], 4),
                       "note": "serving loop through the public API: every step copies q, "
                               "the new tokens' K/V rows and slots, block table and lengths "
                               "from pinned host memory in one packed copy, writes the new "
                               "rows into the resident cache (pattn_reshape_and_cache), runs "
                               "attention and reads the output back; two slots, so a step's "
                               "copies overlap the neighbouring steps' compute (time = "
                               "span of K steps / K)"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(res["case"], spec, counts, pk, args)
    return line


def cpu_baseline(case, spec, counts, pk, args):
    """The float64 oracle as it stands, on the host cores, on a uniform sample
    of the workload sized to ~15 s, in the metric's unit (the sample's share of
    the step's roofline time over the oracle's time); plus a 1-thread time on
    a smaller sample."""
    stride = oracle_stride(case, spec, args.cpu_seconds)
    ob = time_oracle(case, spec, stride)
    frac = ob["row_keys"] / counts["row_keys"]
    t_roof = roofline_seconds(counts, pk) * frac
    one_stride = oracle_stride(case, spec, args.cpu_seconds / 4, threads=1)
    o1 = time_oracle(case, spec, one_stride, threads=1)
    t1_roof = roofline_seconds(counts, pk) * (o1["row_keys"] / counts["row_keys"])
    return {"value": round(100.0 * t_roof / ob["seconds"], 9), "unit": UNIT,
            "cores": ob["cores"], "kind": "oracle", "sample": ob["sample"],
            "seconds": round(ob["seconds"], 3),
            "row_keys_per_s": round(ob["row_keys"] / ob["seconds"], 1),
            "cpu_model": cpu_model(),
            "one_thread": {"value": round(100.0 * t1_roof / o1["seconds"], 9),
                           "seconds": round(o1["seconds"], 3), "cores": 1,
                           "row_keys_per_s": round(o1["row_keys"] / o1["seconds"], 1),
                           "sample": o1["sample"]}}


def run_reference(args, spec, world, rank):
    """The float64 CPU oracle, timed on the host cores (rank 0 only), each step
    a uniform sample of the workload sized so the whole run takes ~2 minutes;
    value in the metric's unit (the sample's share of the step's roofline time
    over the oracle's time)."""
    if world > 1 and rank != 0:
        return 0
    import workloads as W
    case = W.make_case(spec, device="cpu")
    counts = work_counts(spec)
    pk, _ = peaks()
    budget = 120.0 / (args.steps + args.warmup)
    stride = oracle_stride(case, spec, budget)
    for _ in range(args.warmup):
        time_oracle(case, spec, stride)
    times, ob = [], None
    for _ in range(args.steps):
        ob = time_oracle(case, spec, stride)
        times.append(ob["seconds"])
    sec = statistics.mean(times)
    t_roof = roofline_seconds(counts, pk) * ob["row_keys"] / counts["row_keys"]
    value = 100.0 * t_roof / sec
    line = {"metric": METRIC, "impl": "reference", "value": round(value, 9), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(spec, args.config, world),
            "cpu_baseline": {"value": round(value, 9), "unit": UNIT, "cores": ob["cores"],
                             "kind": "oracle", "sample": ob["sample"],
                             "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 9), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main() or 0)
