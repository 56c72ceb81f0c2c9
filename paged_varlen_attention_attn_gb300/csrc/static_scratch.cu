// static_scratch.cu -- split-KV decode that needs no caller workspace.
//
// pattn_varlen_fwd asks its caller for a device workspace.  Some callers have
// none to give and cannot make one: a plugin loaded into a host application
// that owns every byte of device memory through its own allocator, or code on
// a latency-critical path where cudaMalloc / cudaFree would synchronise the
// device.  pattn_decode_fwd_static serves the decode rows of a batch for them:
// the partition partials and the status word live in a file-scope device
// array of fixed size instead, so the call allocates nothing (no cudaMalloc,
// no cudaFree, no allocating library routine).
//
// The array is part of the library's module: every GPU that loads the
// library holds it until the process exits.  Every call shares it and it
// keeps the previous call's contents; the status word is cleared on the
// stream at the start of each call, and every partial the combine step reads
// is written earlier in the same call.  Calls whose work overlaps on the GPU
// (other streams, other host threads) race on the array and must be
// serialised by the caller.
#include <cmath>

#include "../../include/pattn.h"
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(PATTN_STATIC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch in the current context.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress (which allocates nothing) on every call, with the
// caller's device current: a context that was reset or replaced (the module
// loaded again, possibly at another address) never sees a stale pointer.
cudaError_t static_scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace pattn

using namespace pattn;

extern "C" pattn_status_t pattn_decode_fwd_static(
    const void* q, const void* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
    const int32_t* query_start_loc, void* out, float scale, int num_heads, int num_kv_heads,
    int head_size, int block_size, int window, int causal, int kv_dtype, const float* kv_scale,
    int num_seqs, int num_tokens, int max_blocks_per_seq, int num_blocks, int max_seq_len,
    int num_splits, void* stream) {
  if (!q || !kv_cache || !block_table || !seq_lens || !query_start_loc || !out)
    return PATTN_ERR_INVALID_ARGUMENT;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
    return PATTN_ERR_INVALID_ARGUMENT;
  if (block_size <= 0 || block_size % 16 != 0) return PATTN_ERR_INVALID_ARGUMENT;
  if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq < 0 || num_blocks < 0 ||
      max_seq_len < 0 || num_splits < 0 || num_splits > PATTN_MAX_SPLITS)
    return PATTN_ERR_INVALID_ARGUMENT;
  if (head_size != 64 && head_size != 128) return PATTN_ERR_UNSUPPORTED;
  if (num_heads / num_kv_heads > 16) return PATTN_ERR_UNSUPPORTED;
  if (!(scale >= 0.f) || std::isinf(scale)) return PATTN_ERR_INVALID_ARGUMENT;
  if (causal != 0 && causal != 1) return PATTN_ERR_INVALID_ARGUMENT;
  if (kv_dtype != PATTN_KV_BF16 && kv_dtype != PATTN_KV_FP8_E4M3 && kv_dtype != PATTN_KV_F16)
    return PATTN_ERR_UNSUPPORTED;
  if (kv_dtype == PATTN_KV_FP8_E4M3 &&
      (!kv_scale || !(kv_scale[0] > 0.f) || !(kv_scale[1] > 0.f) || std::isinf(kv_scale[0]) ||
       std::isinf(kv_scale[1])))
    return PATTN_ERR_INVALID_ARGUMENT;
  if (!causal && window > 0) return PATTN_ERR_UNSUPPORTED;
  if (window < 0) window = 0;
  if ((reinterpret_cast<uintptr_t>(kv_cache) & 15) || (reinterpret_cast<uintptr_t>(q) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 15))
    return PATTN_ERR_INVALID_ARGUMENT;
  if (num_seqs == 0 || num_tokens == 0) return PATTN_OK;
  if (num_blocks == 0 || max_blocks_per_seq == 0) return PATTN_ERR_INVALID_ARGUMENT;

  // Same partition count as pattn_varlen_fwd would use for these sizes.
  pattn_ext_t ext = {};
  ext.struct_size = sizeof(pattn_ext_t);
  ext.num_seqs = num_seqs;
  ext.num_tokens = num_tokens;
  ext.max_blocks_per_seq = max_blocks_per_seq;
  ext.num_blocks = num_blocks;
  ext.max_query_len = 1;
  ext.max_seq_len = max_seq_len;
  ext.num_splits = num_splits;
  const int splits = pattn_decode_splits(&ext, num_heads, num_kv_heads, block_size, window);
  if (splits < 1) return PATTN_ERR_INVALID_ARGUMENT;
  const WsLayout L = workspace_layout(num_seqs, num_tokens, num_heads, num_kv_heads, head_size, 1,
                                      splits);
  if (L.total > kStaticScratchBytes) return PATTN_ERR_WORKSPACE_TOO_SMALL;

  void* scratch = nullptr;
  if (static_scratch_address(&scratch) != cudaSuccess) return PATTN_ERR_CUDA;
  unsigned char* ws = static_cast<unsigned char*>(scratch);

  Problem p = {};
  p.q = q;
  p.kv = kv_cache;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.out = out;
  p.scale = scale;
  p.H = num_heads;
  p.Hkv = num_kv_heads;
  p.G = num_heads / num_kv_heads;
  p.D = head_size;
  p.bs = block_size;
  p.bs_shift = (block_size & (block_size - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(block_size)) : -1;
  p.window = window;
  p.causal = causal;
  p.kv_dtype = kv_dtype;
  p.k_scale = (kv_dtype == PATTN_KV_FP8_E4M3) ? kv_scale[0] : 1.f;
  p.v_scale = (kv_dtype == PATTN_KV_FP8_E4M3) ? kv_scale[1] : 1.f;
  p.B = num_seqs;
  p.T = num_tokens;
  p.mbps = max_blocks_per_seq;
  p.bt_stride = p.mbps;
  p.kv_chunks = 1;
  p.clear_status = 1;
  p.o32 = nullptr;
  p.lse32 = nullptr;
  p.NB = num_blocks;
  p.max_q = 1;
  // Rows of requests with query_len != 1 are another call's: the kernel leaves
  // them as they are.
  p.decode_rows_only = 1;
  p.max_s = max_seq_len;
  p.splits = splits;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.tiles = nullptr;
  p.max_tiles = 0;
  p.rows_per_item = prefill_rows_per_item(p.G);
  p.counters = reinterpret_cast<unsigned*>(ws + L.counters_off);
  p.o_part = reinterpret_cast<float*>(ws + L.o_part_off);
  p.lse_part = reinterpret_cast<float*>(ws + L.lse_off);
  p.stream = static_cast<cudaStream_t>(stream);

  // The status word and the partition counters must start at zero; the
  // partials need no clearing.
  if (cudaMemsetAsync(ws, 0, L.counters_end, p.stream) != cudaSuccess) return PATTN_ERR_CUDA;
  CUtensorMap dmap;
  if (!encode_decode_map(&dmap, kv_cache, kv_dtype, head_size, num_kv_heads, block_size,
                         num_blocks, decode_heads_per_cta(num_kv_heads, head_size, kv_dtype)))
    return PATTN_ERR_CUDA;
  if (launch_decode(p, dmap) != cudaSuccess) return PATTN_ERR_CUDA;
  return PATTN_OK;
}
