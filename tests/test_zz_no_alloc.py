"""The workspace-free decode entry point, pattn_decode_fwd_static.

It serves callers that cannot allocate device memory or hand over a workspace
(a plugin whose host application owns every byte of device memory, or a
latency-critical path where cudaMalloc / cudaFree would synchronise the
device).  Its scratch lives in a fixed device array inside the library.  These
tests call it through the C ABI: twice in a row on different batches, each
result checked against pattn_varlen_fwd on the same inputs with the
tolerances the parity tests use; on a batch that mixes prefills and decodes,
where the decode rows must match the float64 oracle and every other row must
be left bit for bit as it was; and on a batch too large for the array, which
must be refused before any GPU work.  The file sorts last so that a run which
stops at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import paged_varlen_attention_attn_gb300 as pa
import workloads as W
from cases import small_spec
from gpu_util import assert_close, oracle_all, run_gpu

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


@pytest.mark.parametrize("splits", [0, 5])
def test_static_scratch_mixed_batch_leaves_other_rows_untouched(splits):
    # prefills, chunked prefills and decodes in one batch; out starts as NaN
    spec = small_spec(4545, H=8, Hkv=2, d=128, bs=16, n_req=12, max_s=900,
                      kinds=("prefill", "decode", "chunk", "decode"))
    case = W.make_case(spec, device=DEV)
    assert any(q == 1 for q in spec.q_lens) and any(q > 1 for q in spec.q_lens)
    out = torch.full_like(case.q, float("nan"))
    before = out.view(torch.int16).cpu().numpy().copy()
    assert call_static(case, splits, out) == 0
    torch.cuda.synchronize()
    got_bits = out.view(torch.int16).cpu().numpy()
    got = out.float().cpu().numpy().astype(np.float64)
    ref, _ = oracle_all(case)
    qsl = case.query_start_loc.cpu().numpy()
    decode_rows = np.zeros(case.num_tokens, dtype=bool)
    for r, ql in enumerate(spec.q_lens):
        if ql == 1:
            decode_rows[int(qsl[r])] = True
    # every row that is not a decode row keeps its bits
    assert np.array_equal(got_bits[~decode_rows], before[~decode_rows])
    # decode rows match the oracle
    assert_close(got[decode_rows], ref[decode_rows], spec.kv_dtype)


def test_static_scratch_rejects_batches_beyond_its_size():
    # 16384 real decode requests (query_len 1, seq_len 16, one block each,
    # all on block 0), so the metadata covers every request the call names:
    # with 64 forced partitions the partials need 16384 x 4 heads x 64 x 65
    # floats, more than the fixed array, and the call must be refused on the
    # host before any GPU work.
    B, H, Hkv, d, bs = 1 << 14, 4, 2, 64, 16
    q = torch.zeros(B, H, d, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros_like(q)
    kv = torch.zeros(2, 1, bs, Hkv, d, dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros(B, 1, dtype=torch.int32, device=DEV)
    seq_lens = torch.full((B,), bs, dtype=torch.int32, device=DEV)
    qsl = torch.arange(B + 1, dtype=torch.int32, device=DEV)
    need = B * H * 64 * (d + 1) * 4
    assert need > pa.STATIC_SCRATCH_BYTES
    st = pa.pattn_decode_fwd_static(
        q.data_ptr(), kv.data_ptr(), bt.data_ptr(), seq_lens.data_ptr(), qsl.data_ptr(),
        out.data_ptr(), 0.125, H, Hkv, d, bs, 0, 1, 0, None, B, B, 1, 1, bs, 64,
        torch.cuda.current_stream().cuda_stream)
    assert st == 3  # PATTN_ERR_WORKSPACE_TOO_SMALL, before any GPU work
