"""The workspace-free decode entry point, pattn_decode_fwd_static.

It serves callers that cannot allocate device memory or hand over a workspace
(a plugin whose host application owns every byte of device memory, or a
latency-critical path where cudaMalloc / cudaFree would synchronise the
device).  Its scratch lives in a fixed device array inside the library.  This
test calls it through the C ABI twice in a row, on different batches, and
checks each result against pattn_varlen_fwd on the same inputs, with the
tolerances the parity tests use.  The file sorts last so that a run which stops
at the first failure has already run every other test.
"""
import pytest
import torch

import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from cases import small_spec
from gpu_util import assert_close, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_varlen_attention_attn_gb300 import _build
    _build.build()
    pa.load()


def call_static(case, num_splits, out):
    s = case.spec
    stream = torch.cuda.current_stream()
    st = pa.pattn_decode_fwd_static(
        case.q.data_ptr(), case.kv_cache.data_ptr(), case.block_table.data_ptr(),
        case.seq_lens.data_ptr(), case.query_start_loc.data_ptr(), out.data_ptr(),
        case.scale, s.num_heads, s.num_kv_heads, s.head_size, s.block_size, s.window,
        s.causal, s.kv_dtype, case.kv_scale if s.kv_dtype else None, case.num_seqs,
        case.num_tokens, case.block_table.shape[1], case.num_blocks, case.max_seq_len,
        num_splits, stream.cuda_stream)
    return st


def test_static_scratch_decode_matches_workspace_path_twice():
    first = W.make_case(small_spec(4242, H=16, Hkv=2, d=128, bs=16, n_req=9, max_s=3000,
                                   kinds=("decode",)), device=DEV)
    second = W.make_case(small_spec(4343, H=32, Hkv=8, d=128, bs=64, n_req=5, max_s=5000,
                                    window=700, kv_dtype=W.KV_FP8_E4M3, kinds=("decode",)),
                         device=DEV)
    results = []
    for case, splits in ((first, 8), (second, 0)):
        out = torch.full_like(case.q, float("nan"))
        assert call_static(case, splits, out) == 0
        results.append(out)
    torch.cuda.synchronize()
    for (case, splits), got in zip(((first, 8), (second, 0)), results):
        ref = run_gpu(case, num_splits=splits)
        assert_close(got.float().cpu().numpy(), ref.float().cpu().numpy().astype("float64"),
                     case.spec.kv_dtype)


def test_static_scratch_rejects_batches_beyond_its_size():
    case = W.make_case(small_spec(4444, H=16, Hkv=2, d=128, bs=16, n_req=2, max_s=200,
                                  kinds=("decode",)), device=DEV)
    out = torch.zeros_like(case.q)
    # 2**14 requests x 16 heads x 64 partitions x 129 floats > the fixed array
    s = case.spec
    st = pa.pattn_decode_fwd_static(
        case.q.data_ptr(), case.kv_cache.data_ptr(), case.block_table.data_ptr(),
        case.seq_lens.data_ptr(), case.query_start_loc.data_ptr(), out.data_ptr(),
        case.scale, s.num_heads, s.num_kv_heads, s.head_size, s.block_size, 0, 1, 0, None,
        1 << 14, case.num_tokens, case.block_table.shape[1], case.num_blocks,
        case.max_seq_len, 64, torch.cuda.current_stream().cuda_stream)
    assert st == 3  # PATTN_ERR_WORKSPACE_TOO_SMALL, before any GPU work
