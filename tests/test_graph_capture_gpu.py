"""A pattn_varlen_fwd call captured in a CUDA graph and replayed with new
batch contents.

The call allocates nothing, never synchronises and reads the batch metadata
(block tables, sequence lengths, query start offsets) on the device, so a
serving loop can capture it once and replay it for every step whose batch fits
the host-side sizes given at capture (number of requests and tokens, the
block-table width, max_query_len, max_seq_len, the partition count).  The test
captures one call, then replays it on two different batches written into the
same buffers and compares each with the float64 oracle."""
import pytest
import torch

import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from gpu_util import assert_close, oracle_all

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
# Host-side bounds baked into the captured call.
MAX_Q, MAX_S = 64, 768


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_varlen_attention_attn_gb300 import _build
    _build.build()
    pa.load()


def _spec(name, seq_lens, seed):
    # same shapes for both batches: 4 requests (a prefill chunk, two decodes,
    # a full prefill), 103 tokens, 48-entry block-table rows, 120-block pool
    q_lens = [64, 1, 1, 37]
    return W.CaseSpec(name, q_lens, seq_lens, 8, 2, 128, 16, pool_blocks=120,
                      max_blocks_per_seq=MAX_S // 16, seed=seed)


def _call(bufs, ws, stream):
    c = bufs
    s = c.spec
    return pa.forward(c.q, c.kv_cache, c.block_table, c.seq_lens, c.query_start_loc,
                      scale=c.scale, num_heads=s.num_heads, num_kv_heads=s.num_kv_heads,
                      head_size=s.head_size, block_size=s.block_size, window=s.window,
                      causal=s.causal, kv_dtype=s.kv_dtype, kv_scale=None,
                      max_query_len=MAX_Q, max_seq_len=MAX_S, out=c.out, workspace=ws,
                      stream=stream)


def _load(bufs, case):
    for name in ("q", "kv_cache", "block_table", "seq_lens", "query_start_loc"):
        getattr(bufs, name).copy_(getattr(case, name))
    bufs.out.fill_(float("nan"))


def _check(bufs, case):
    st = pa.pattn_read_device_status(pa.forward.last_ext)
    assert st == 0, pa.pattn_status_string(st)
    ref, _ = oracle_all(case)
    assert_close(bufs.out.float().cpu().numpy(), ref, case.spec.kv_dtype)


def test_captured_call_replays_on_new_batches():
    a = W.make_case(_spec("graph_a", [300, 700, 129, 37], 1101), device=DEV)
    b = W.make_case(_spec("graph_b", [100, 500, 760, 40], 1102), device=DEV)
    bufs = W.make_case(_spec("graph_bufs", [300, 700, 129, 37], 1101), device=DEV)
    bufs.out = torch.empty_like(bufs.q)
    ws = pa.Workspace()
    stream = torch.cuda.Stream(DEV)

    # eager call first: sizes the workspace and does the library's one-time set-up
    _load(bufs, a)
    with torch.cuda.stream(stream):
        _call(bufs, ws, stream)
    torch.cuda.synchronize()
    _check(bufs, a)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        _call(bufs, ws, torch.cuda.current_stream())
    torch.cuda.synchronize()

    for case in (b, a, b):
        _load(bufs, case)
        graph.replay()
        torch.cuda.synchronize()
        _check(bufs, case)
