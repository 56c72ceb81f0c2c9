"""Host-side checks of bench.py: the algorithmic work counters, the
world-size-2 aggregation (gloo, CPU), and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _brute_visible(spec):
    dec = pre = 0
    for ql, s in zip(spec.q_lens, spec.seq_lens):
        for i in range(ql):
            p = s - ql + i
            n = sum(1 for k in range(s) if (not spec.causal or k <= p)
                    and (spec.window <= 0 or p - k < spec.window))
            if ql == 1:
                dec += n
            else:
                pre += n
    return dec, pre


@pytest.mark.parametrize("window,causal", [(0, 1), (5, 1), (0, 0)])
def test_work_counts_match_a_direct_count(window, causal):
    spec = W.CaseSpec("c", [1, 7, 1, 30], [40, 50, 3, 30], 4, 2, 64, 16, window=window,
                      causal=causal)
    dec, pre = _brute_visible(spec)
    c = bench.work_counts(spec)
    assert c["flops_prefill"] == 4.0 * 64 * 4 * pre
    assert c["bytes_decode"] == dec * 2 * 2 * 64 * 2
    assert c["tokens"] == 39


def test_config_counts_match_the_survey_figures():
    c2 = bench.work_counts(W.config_spec(2))
    assert 0.4e9 < c2["bytes_decode"] < 0.8e9          # ~0.6 GB of visible KV
    c5 = bench.work_counts(W.config_spec(5))
    assert c5["bytes_decode"] == 8 * 131072 * 2 * 8 * 128
    c4 = bench.work_counts(W.config_spec(4))
    assert c4["flops_prefill"] == 4 * 2048 * 4096 * 4 * 128 * 64


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init("gloo")
    units = [3.0, 5.0][rank]
    secs = [0.5, 2.0][rank]
    v, slowest = bench.aggregate(units, secs)
    q.put((rank, v, slowest))
    bench.barrier()
    torch.distributed.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, v, slowest in got:
        assert slowest == 2.0 and v == pytest.approx(8.0 / 2.0)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "1", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    # the same metric, unit and config as the GPU arm's line for this workload
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["config"] == bench.config_dict(W.config_spec(1), 1, 1)


def test_oracle_sample_counts_visible_pairs():
    # the sampled (row, key) count is what the oracle's loops visit: checked
    # against a direct count on the mixed workload's lengths
    spec = W.config_spec(1)
    case = W.make_case(spec, device="cpu")
    smp = bench.oracle_sample(case, spec, 1)
    rk = bench.sample_row_keys(spec, smp["qsl"], smp["rows"])
    assert rk == bench.work_counts(spec)["row_keys"]
    assert rk == spec.num_heads * (sum(range(1, 9)) + 40)
