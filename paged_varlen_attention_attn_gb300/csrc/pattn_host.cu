// pattn_host.cu -- the C ABI of libpattn (declared in include/pattn.h).
//
// Host work per call: check the host-side arguments (returning a status before
// any CUDA call), lay out the caller's workspace, encode the two TMA tensor
// maps, and enqueue plan -> prefill -> decode -> combine on the caller's
// stream.  Nothing here synchronises or allocates.
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/pattn.h"
#include "common.cuh"
#include "internal.h"

namespace pattn {

namespace {

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Number of SMs of the current device (cached per device).
int sm_count() {
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    counts[dev] = n;
  }
  return counts[dev];
}

bool ext_ok(const pattn_ext_t* ext) {
  return ext && ext->struct_size >= sizeof(pattn_ext_t);
}

// Decode partition count.  A forced count is used as given; otherwise enough
// partitions that there are about 8 (request, KV head, partition) items per
// SM (2 to 4 decode CTAs, depending on how many KV heads one CTA serves), and
// that no partition is longer than ~1024 keys, bounded by the block count a
// row can see and by PATTN_MAX_SPLITS.  It depends on neither dtype nor head
// size, so pattn_workspace_bytes can size the partials without them.
int choose_splits(const pattn_ext_t* ext, int num_kv_heads, int block_size, int window) {
  if (ext->num_splits > 0) return ext->num_splits;
  const int visible = (window > 0) ? std::min(ext->max_seq_len, window + block_size)
                                   : ext->max_seq_len;
  const int max_blocks = std::max(1, (visible + block_size - 1) / block_size);
  const long long items = static_cast<long long>(std::max(1, ext->num_seqs)) * num_kv_heads;
  const int sms = sm_count();
  int by_grid = static_cast<int>((8LL * sms + items - 1) / items);
  int by_len = (visible + 1023) / 1024;
  int s = std::max(1, std::max(by_grid, by_len));
  s = std::min(s, max_blocks);
  s = std::min(s, PATTN_MAX_SPLITS);
  return std::max(1, s);
}

pattn_status_t validate(const pattn_ext_t* ext, int num_heads, int num_kv_heads, int head_size,
                        int block_size) {
  if (!ext_ok(ext)) return PATTN_ERR_INVALID_ARGUMENT;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0)
    return PATTN_ERR_INVALID_ARGUMENT;
  if (block_size <= 0 || block_size % 16 != 0) return PATTN_ERR_INVALID_ARGUMENT;
  if (ext->num_seqs < 0 || ext->num_tokens < 0 || ext->max_blocks_per_seq < 0 ||
      ext->num_blocks < 0 || ext->max_query_len < 0 || ext->max_seq_len < 0 ||
      ext->num_splits < 0 || ext->num_splits > PATTN_MAX_SPLITS)
    return PATTN_ERR_INVALID_ARGUMENT;
  if (head_size != 64 && head_size != 128) return PATTN_ERR_UNSUPPORTED;
  if (num_heads / num_kv_heads > 16) return PATTN_ERR_UNSUPPORTED;
  return PATTN_OK;
}

}  // namespace

bool encode_kv_map(CUtensorMap* map, const void* kv_cache, int kv_dtype, int D, int Hkv, int bs,
                   int NB, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const bool fp8 = kv_dtype == PATTN_KV_FP8_E4M3;
  const cuuint64_t es = fp8 ? 1 : 2;
  const cuuint64_t row = static_cast<cuuint64_t>(D) * es;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(bs), 2ull * static_cast<cuuint64_t>(NB)};
  cuuint64_t strides[3] = {row, row * Hkv, row * Hkv * bs};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(fp8 ? D : 64), 1,
                       static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw =
      (fp8 && D == 64) ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  return enc(map,
             fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                 : (kv_dtype == PATTN_KV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16),
             4,
             const_cast<void*>(kv_cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_decode_map(CUtensorMap* map, const void* kv_cache, int kv_dtype, int D, int Hkv,
                       int bs, int NB, int heads) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  if (kv_dtype == PATTN_KV_FP8_E4M3) {
    const cuuint64_t row = static_cast<cuuint64_t>(D);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(bs),
                          static_cast<cuuint64_t>(Hkv), 2ull * static_cast<cuuint64_t>(NB)};
    cuuint64_t strides[3] = {row * Hkv, row, row * Hkv * bs};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(D), 16, static_cast<cuuint32_t>(heads), 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(kv_cache), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               D == 64 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t row = static_cast<cuuint64_t>(D) * 2;
  cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(bs), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(D / 64), 2ull * static_cast<cuuint64_t>(NB)};
  cuuint64_t strides[4] = {row * Hkv, row, 128, row * Hkv * bs};
  cuuint32_t box[5] = {64, 16, static_cast<cuuint32_t>(heads), static_cast<cuuint32_t>(D / 64), 1};
  return enc(map,
             kv_dtype == PATTN_KV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
             5, const_cast<void*>(kv_cache), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

WsLayout workspace_layout(int B, int T, int H, int Hkv, int D, int max_q, int splits) {
  WsLayout L;
  size_t off = sizeof(WsHeader);
  L.counters_off = off;
  L.counters_end = off + static_cast<size_t>(B) * Hkv * sizeof(unsigned);
  off = align_up(L.counters_end, 256);
  L.max_tiles = (max_q > 1) ? (T + BLOCK_M - 1) / BLOCK_M + B : 0;
  L.tiles_off = off;
  off = align_up(off + static_cast<size_t>(L.max_tiles) * sizeof(int2), 256);
  L.o_part_off = off;
  if (splits > 1) {
    off = align_up(off + static_cast<size_t>(B) * H * splits * D * sizeof(float), 256);
    L.lse_off = off;
    off = align_up(off + static_cast<size_t>(B) * H * splits * sizeof(float), 256);
  } else {
    L.lse_off = off;
  }
  L.total = off;
  return L;
}

}  // namespace pattn

using namespace pattn;

extern "C" {

int pattn_version(void) { return 10000; }

const char* pattn_status_string(int s) {
  switch (s) {
    case PATTN_OK: return "ok";
    case PATTN_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case PATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PATTN_ERR_CUDA: return "CUDA error";
    case PATTN_ERR_BAD_METADATA: return "bad metadata detected on the device";
    case PATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int pattn_decode_splits(const pattn_ext_t* ext, int num_heads, int num_kv_heads, int block_size,
                        int window) {
  if (validate(ext, num_heads, num_kv_heads, 128, block_size) != PATTN_OK) return 0;
  return choose_splits(ext, num_kv_heads, block_size, window);
}

size_t pattn_workspace_bytes(const pattn_ext_t* ext, int num_heads, int num_kv_heads,
                             int head_size, int block_size) {
  if (validate(ext, num_heads, num_kv_heads, head_size, block_size) != PATTN_OK) return 0;
  // The window only lowers the automatic split count; size for no window.
  const int splits = choose_splits(ext, num_kv_heads, block_size, 0);
  return workspace_layout(ext->num_seqs, ext->num_tokens, num_heads, num_kv_heads, head_size,
                          ext->max_query_len, splits)
      .total;
}

pattn_status_t pattn_read_device_status(const pattn_ext_t* ext) {
  if (!ext_ok(ext) || !ext->workspace) return PATTN_ERR_INVALID_ARGUMENT;
  cudaStream_t st = static_cast<cudaStream_t>(ext->stream);
  unsigned host = 0;
  WsHeader* hdr = static_cast<WsHeader*>(ext->workspace);
  if (cudaMemcpyAsync(&host, &hdr->status, sizeof(unsigned), cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return PATTN_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PATTN_ERR_CUDA;
  if (cudaMemsetAsync(&hdr->status, 0, sizeof(unsigned), st) != cudaSuccess) return PATTN_ERR_CUDA;
  if (host & PATTN_DEV_TIMEOUT) return PATTN_ERR_DEVICE_TIMEOUT;
  if (host & PATTN_DEV_BAD_METADATA) return PATTN_ERR_BAD_METADATA;
  return PATTN_OK;
}

pattn_status_t pattn_varlen_fwd(const void* q, const void* kv_cache, const int32_t* block_table,
                                const int32_t* seq_lens, const int32_t* query_start_loc,
                                void* out, float scale, int num_heads, int num_kv_heads,
                                int head_size, int block_size, int window, int causal,
                                int kv_dtype, const float* kv_scale, const pattn_ext_t* ext) {
  pattn_status_t v = validate(ext, num_heads, num_kv_heads, head_size, block_size);
  if (v != PATTN_OK) return v;
  if (!q || !kv_cache || !block_table || !seq_lens || !query_start_loc || !out || !ext->workspace)
    return PATTN_ERR_INVALID_ARGUMENT;
  if (!(scale >= 0.f) || std::isinf(scale)) return PATTN_ERR_INVALID_ARGUMENT;
  if (causal != 0 && causal != 1) return PATTN_ERR_INVALID_ARGUMENT;
  if (kv_dtype != PATTN_KV_BF16 && kv_dtype != PATTN_KV_FP8_E4M3 && kv_dtype != PATTN_KV_F16)
    return PATTN_ERR_UNSUPPORTED;
  if (kv_dtype == PATTN_KV_FP8_E4M3) {
    if (!kv_scale || !(kv_scale[0] > 0.f) || !(kv_scale[1] > 0.f) || std::isinf(kv_scale[0]) ||
        std::isinf(kv_scale[1]))
      return PATTN_ERR_INVALID_ARGUMENT;
  }
  if (!causal && window > 0) return PATTN_ERR_UNSUPPORTED;
  if (window < 0) window = 0;
  if (kv_dtype == PATTN_KV_FP8_E4M3 && ext->max_query_len > 1) return PATTN_ERR_UNSUPPORTED;
  // Prefill key tiles are 128 keys: a page must divide the tile or be a whole
  // number of tiles.
  if (ext->max_query_len > 1 && !(BLOCK_N % block_size == 0 || block_size % BLOCK_N == 0))
    return PATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(kv_cache) & 15) || (reinterpret_cast<uintptr_t>(q) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 15) ||
      (reinterpret_cast<uintptr_t>(ext->workspace) & 255))
    return PATTN_ERR_INVALID_ARGUMENT;

  const int splits = choose_splits(ext, num_kv_heads, block_size, window);
  const WsLayout L = workspace_layout(ext->num_seqs, ext->num_tokens, num_heads, num_kv_heads, head_size,
                                      ext->max_query_len, splits);
  if (ext->workspace_bytes < L.total) return PATTN_ERR_WORKSPACE_TOO_SMALL;
  if (ext->num_seqs == 0 || ext->num_tokens == 0) return PATTN_OK;
  if (ext->num_blocks == 0 || ext->max_blocks_per_seq == 0) return PATTN_ERR_INVALID_ARGUMENT;

  Problem p;
  std::memset(&p, 0, sizeof p);
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
  p.B = ext->num_seqs;
  p.T = ext->num_tokens;
  p.mbps = ext->max_blocks_per_seq;
  p.NB = ext->num_blocks;
  p.max_q = ext->max_query_len;
  p.max_s = ext->max_seq_len;
  p.splits = splits;
  unsigned char* ws = static_cast<unsigned char*>(ext->workspace);
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.tiles = reinterpret_cast<int2*>(ws + L.tiles_off);
  p.max_tiles = L.max_tiles;
  p.rows_per_item = prefill_rows_per_item(p.G);
  p.counters = reinterpret_cast<unsigned*>(ws + L.counters_off);
  p.o_part = reinterpret_cast<float*>(ws + L.o_part_off);
  p.lse_part = reinterpret_cast<float*>(ws + L.lse_off);
  p.stream = static_cast<cudaStream_t>(ext->stream);

  // Optional per-phase events (profiling): [2k] before and [2k+1] after phase k.
  auto mark = [&](int idx) {
    if (ext->timing_events && ext->timing_events[idx])
      cudaEventRecord(static_cast<cudaEvent_t>(ext->timing_events[idx]), p.stream);
  };

  mark(0);
  if (ext->max_query_len > 1) {
    // The plan kernel clears the header and the counters and builds the
    // prefill work list.
    if (launch_plan(p) != cudaSuccess) return PATTN_ERR_CUDA;
  } else {
    // Decode only: nothing to plan (the decode kernel validates its own
    // rows); clear the status word and the partition counters.
    if (cudaMemsetAsync(ws, 0, L.counters_end, p.stream) != cudaSuccess) return PATTN_ERR_CUDA;
  }
  mark(1);
  mark(2);

  if (ext->max_query_len > 1) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PATTN_ERR_CUDA;
    CUtensorMap qmap, kvmap;
    const cuuint64_t es = 2;
    {
      cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_size),
                            static_cast<cuuint64_t>(num_heads),
                            static_cast<cuuint64_t>(ext->num_tokens)};
      cuuint64_t strides[2] = {head_size * es, static_cast<cuuint64_t>(num_heads) * head_size * es};
      cuuint32_t box[3] = {64, 1, BLOCK_M};
      cuuint32_t estr[3] = {1, 1, 1};
      const CUtensorMapDataType qt = (kv_dtype == PATTN_KV_F16) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      if (enc(&qmap, qt, 3, const_cast<void*>(q), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PATTN_ERR_CUDA;
    }
    if (!encode_kv_map(&kvmap, kv_cache, kv_dtype, head_size, num_kv_heads, block_size,
                       ext->num_blocks, std::min(block_size, BLOCK_N)))
      return PATTN_ERR_CUDA;
    if (launch_prefill(p, qmap, kvmap) != cudaSuccess) return PATTN_ERR_CUDA;
  }
  mark(3);
  mark(4);
  CUtensorMap dmap;
  if (!encode_decode_map(&dmap, kv_cache, kv_dtype, head_size, num_kv_heads, block_size,
                         ext->num_blocks, decode_heads_per_cta(num_kv_heads, head_size, kv_dtype)))
    return PATTN_ERR_CUDA;
  if (launch_decode(p, dmap) != cudaSuccess) return PATTN_ERR_CUDA;
  mark(5);
  // The partitions are merged inside the decode kernel (its last CTA of each
  // request and KV-head group); the combine phase is empty.
  mark(6);
  mark(7);
  return PATTN_OK;
}

}  // extern "C"
