// pattn_host.cu -- the C ABI of libpattn (declared in include/pattn.h).
//
// Host work per call: check the host-side arguments (returning a status before
// any CUDA call), lay out the caller's workspace, encode the two TMA tensor
// maps, and enqueue plan -> prefill -> decode -> combine on the caller's
// stream.  Nothing here synchronises or allocates.
#include <cmath>
#include <cstddef>
#include <cstring>
#include <atomic>
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

// The struct grows at its end: a struct_size that reaches the field before
// `sinks` is a complete older struct.
bool ext_ok(const pattn_ext_t* ext) {
  return ext && ext->struct_size >= offsetof(pattn_ext_t, sinks);
}

// ext->sinks if the caller's struct has the field, else null.
const float* ext_sinks(const pattn_ext_t* ext) {
  return ext->struct_size >= offsetof(pattn_ext_t, sinks) + sizeof(ext->sinks) ? ext->sinks
                                                                               : nullptr;
}

// ext->head_size_v if the caller's struct has the field, else 0.
int ext_head_size_v(const pattn_ext_t* ext) {
  return ext->struct_size >= offsetof(pattn_ext_t, head_size_v) + sizeof(ext->head_size_v)
             ? ext->head_size_v
             : 0;
}

// Decode partition count.  A forced count is used as given; otherwise enough
// partitions that there are about 7 (request, KV head, partition) items per
// SM, rounded down (about two decode CTAs per SM, depending on how many KV
// heads one CTA serves), and that no partition is longer than ~8192 keys,
// bounded by the block count a row can see and by PATTN_MAX_SPLITS.  The decode grid runs the requests
// longest first, so its ragged end is short partitions and few, long
// partitions beat many short ones (each CTA has a fixed set-up and merge
// cost); the length bound only keeps one very long request from becoming the
// tail.  It depends on neither dtype nor head size, so pattn_workspace_bytes
// can size the partials without them.
int choose_splits(const pattn_ext_t* ext, int num_kv_heads, int block_size, int window) {
  if (ext->num_splits > 0) return ext->num_splits;
  const int visible = (window > 0) ? std::min(ext->max_seq_len, window + block_size)
                                   : ext->max_seq_len;
  const int max_blocks = std::max(1, (visible + block_size - 1) / block_size);
  const long long items = static_cast<long long>(std::max(1, ext->num_seqs)) * num_kv_heads;
  const int sms = sm_count();
  int by_grid = static_cast<int>(7LL * sms / items);
  int by_len = (visible + 8191) / 8192;
  int s = std::max(1, std::max(by_grid, by_len));
  s = std::min(s, max_blocks);
  s = std::min(s, PATTN_MAX_SPLITS);
  return std::max(1, s);
}

pattn_status_t validate(const pattn_ext_t* ext, int num_heads, int num_kv_heads, int head_size,
                        int block_size);

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
  const int hv = ext_head_size_v(ext);
  if (hv < 0) return PATTN_ERR_INVALID_ARGUMENT;
  if (hv > 0) {  // DiffKV: the generic kernel's sizes
    if (head_size % 32 || head_size < 32 || head_size > 256 || hv % 32 || hv > 256)
      return PATTN_ERR_UNSUPPORTED;
  } else if (head_size != 64 && head_size != 128) {
    return PATTN_ERR_UNSUPPORTED;
  }
  if (num_heads / num_kv_heads > 16) return PATTN_ERR_UNSUPPORTED;
  return PATTN_OK;
}

// Argument checks shared by pattn_varlen_fwd and pattn_cascade_fwd (host
// only, before any CUDA call).
pattn_status_t check_call(const void* q, const void* kv_cache, const int32_t* block_table,
                          const int32_t* seq_lens, const int32_t* query_start_loc, void* out,
                          float scale, int num_heads, int num_kv_heads, int head_size,
                          int block_size, int window, int causal, int kv_dtype,
                          const float* kv_scale, const pattn_ext_t* ext) {
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
  if (ext_head_size_v(ext) > 0 && kv_dtype == PATTN_KV_FP8_E4M3) return PATTN_ERR_UNSUPPORTED;
  // Prefill key tiles of the tensor-core kernel are 128 keys: a page must
  // divide the tile or be a whole number of tiles.
  if (ext->max_query_len > 1 && !(BLOCK_N % block_size == 0 || block_size % BLOCK_N == 0))
    return PATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(kv_cache) & 15) || (reinterpret_cast<uintptr_t>(q) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 15) ||
      (reinterpret_cast<uintptr_t>(ext->workspace) & 255))
    return PATTN_ERR_INVALID_ARGUMENT;
  return PATTN_OK;
}

// Cost model of the co-scheduled mixed batch (measured on GB300): a prefill
// key tile of one item (two 128-row sub-tiles, 128 keys) takes about
// 2.1 us per SM at head size 128 (about 1.3 us at 64; e4m3 tiles 1.1-1.4x
// longer, for the widening: 1.3x is taken, and the mixed step's time was the
// same for 0.95x to 1.3x); beside the prefill, one SM running two decode
// CTAs streams about 120 GB/s of 16-bit K/V (e4m3 about 100 GB/s); decode
// gets about 85 % of HBM beside the prefill.  (A sweep of the prefill grid
// on the mixed workload put the best at 128 of 152 SMs, which these figures
// reproduce.)  The estimate only balances the two kernels; the result does
// not depend on it.
void set_cost_model(Problem& p) {
  p.num_sms = sm_count();
  const bool fp8 = p.kv_dtype == PATTN_KV_FP8_E4M3;
  p.pf_us_per_tile = (p.D == 128 ? 2.1f : 1.3f) * (fp8 ? 1.3f : 1.f);
  p.dec_bytes_per_us = fp8 ? 100000.f : 120000.f;
  p.hbm_bytes_per_us = 0.85f * 6800000.f;
}

// The fields of a Problem every pass shares.
void base_problem(Problem& p, const void* q, const void* kv_cache, void* out, float scale,
                  int num_heads, int num_kv_heads, int head_size, int block_size, int kv_dtype,
                  const float* kv_scale, const pattn_ext_t* ext) {
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.kv = kv_cache;
  p.out = out;
  p.scale = scale;
  p.H = num_heads;
  p.Hkv = num_kv_heads;
  p.G = num_heads / num_kv_heads;
  p.D = head_size;
  p.bs = block_size;
  p.bs_shift = (block_size & (block_size - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(block_size)) : -1;
  p.kv_dtype = kv_dtype;
  p.k_scale = (kv_dtype == PATTN_KV_FP8_E4M3) ? kv_scale[0] : 1.f;
  p.v_scale = (kv_dtype == PATTN_KV_FP8_E4M3) ? kv_scale[1] : 1.f;
  p.T = ext->num_tokens;
  p.NB = ext->num_blocks;
  p.rows_per_item = prefill_rows_per_item(p.G);
  p.kv_chunks = 1;
  p.stream = static_cast<cudaStream_t>(ext->stream);
}

// TMA tensor map over q [T][H][D] with 128-row x 64-element boxes.
bool encode_q_map(CUtensorMap* map, const void* q, int kv_dtype, int H, int D, int T) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t es = 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {D * es, static_cast<cuuint64_t>(H) * D * es};
  cuuint32_t box[3] = {64, 1, BLOCK_M};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType qt = (kv_dtype == PATTN_KV_F16) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return enc(map, qt, 3, const_cast<void*>(q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The prefill kernel (when the pass has rows with query_len > 1), then the
// decode kernel, for one pass.
pattn_status_t launch_pass(const Problem& p) {
  if (p.max_q > 1) {
    CUtensorMap qmap, kmap, vmap;
    if (!encode_prefill_maps(&qmap, &kmap, &vmap, p.q, p.kv, p.kv_dtype, p.H, p.D, p.T, p.Hkv,
                             p.bs, p.NB))
      return PATTN_ERR_CUDA;
    if (launch_prefill(p, qmap, kmap, vmap) != cudaSuccess) return PATTN_ERR_CUDA;
  }
  CUtensorMap dmap;
  if (!encode_decode_map(&dmap, p.kv, p.kv_dtype, p.D, p.Hkv, p.bs, p.NB,
                         decode_heads_per_cta(p.Hkv, p.D, p.kv_dtype)))
    return PATTN_ERR_CUDA;
  if (launch_decode(p, dmap) != cudaSuccess) return PATTN_ERR_CUDA;
  return PATTN_OK;
}

// Workspace of a cascade call: the suffix pass's layout (its header holds the
// call's status word), the prefix pass's, the two passes' fp32 partial
// results, and the passes' metadata (prefix qsl[2] and seq_len, suffix
// seq_lens[B]).
struct CascadeLayout {
  WsLayout suf, pre;
  int splits_suf, splits_pre;
  int kc;  // key chunks of the prefix pass (its prefill CTAs per row item)
  size_t pre_off, o_pre, lse_pre, o_suf, lse_suf, meta, total;
};

CascadeLayout cascade_layout(const pattn_ext_t* ext, int H, int Hkv, int D, int bs, int prefix) {
  CascadeLayout c;
  pattn_ext_t es = *ext;
  es.max_seq_len = std::max(1, ext->max_seq_len - prefix);
  pattn_ext_t ep = *ext;
  ep.num_seqs = 1;
  ep.max_query_len = ext->num_tokens;
  ep.max_seq_len = prefix;
  c.splits_suf = choose_splits(&es, Hkv, bs, 0);
  c.splits_pre = choose_splits(&ep, Hkv, bs, 0);
  c.suf = workspace_layout(ext->num_seqs, ext->num_tokens, H, Hkv, D, ext->max_query_len,
                           c.splits_suf);
  c.pre = workspace_layout(1, ext->num_tokens, H, Hkv, D, ext->num_tokens, c.splits_pre);
  // Key chunks for the prefix pass: enough prefill CTAs for ~2 per SM when
  // the batch has few query rows (one 128-row tile per head pair otherwise
  // walks the whole prefix alone), at most one per key tile and at most 16.
  {
    const int G = H / Hkv;
    const long long items = static_cast<long long>((ext->num_tokens + prefill_rows_per_item(G) - 1) /
                                                   prefill_rows_per_item(G)) *
                            ((G % 2 == 0) ? H / 2 : H);
    const long long want = (2LL * sm_count() + items - 1) / std::max(1LL, items);
    long long kc = std::min(want, 16LL);
    kc = std::min(kc, static_cast<long long>((prefix + BLOCK_N - 1) / BLOCK_N));
    c.kc = static_cast<int>(std::max(1LL, kc));
  }
  const size_t rows = static_cast<size_t>(ext->num_tokens) * H;
  size_t off = align_up(c.suf.total, 256);
  c.pre_off = off;
  off = align_up(off + c.pre.total, 256);
  c.o_pre = off;
  off = align_up(off + rows * c.kc * D * sizeof(float), 256);
  c.lse_pre = off;
  off = align_up(off + rows * c.kc * sizeof(float), 256);
  c.o_suf = off;
  off = align_up(off + rows * D * sizeof(float), 256);
  c.lse_suf = off;
  off = align_up(off + rows * sizeof(float), 256);
  c.meta = off;
  off = align_up(off + (3 + static_cast<size_t>(ext->num_seqs)) * sizeof(int), 256);
  c.total = off;
  return c;
}


}  // namespace

#ifdef PATTN_WAIT_TEST
namespace {
std::atomic<int> g_test_wait_skip{0};
}
int test_wait_skip() { return g_test_wait_skip.load(); }
#endif

bool encode_kv_map(CUtensorMap* map, const void* kv_cache, int kv_dtype, int D, int Hkv, int bs,
                   int NB, int box_rows, bool v_groups) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  if (kv_dtype == PATTN_KV_FP8_E4M3) {
    // e4m3 rows: for the prefill kernel's 8-bit score MMAs (d 128, v_groups
    // false) in the 128-byte-swizzled K-major layout; otherwise unswizzled,
    // into the ring stage where the producers widen them to the swizzled f16
    // layout.
    const bool sw = !v_groups && D == 128;
    const cuuint64_t row = static_cast<cuuint64_t>(D);
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                          static_cast<cuuint64_t>(bs), 2ull * static_cast<cuuint64_t>(NB)};
    cuuint64_t strides[3] = {row, row * Hkv, row * Hkv * bs};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(D), 1, static_cast<cuuint32_t>(box_rows), 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(kv_cache), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               sw ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t row = static_cast<cuuint64_t>(D) * 2;
  const CUtensorMapDataType dt = kv_dtype == PATTN_KV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (v_groups) {
    // {64, row of a 16-slot group, d half, head, group}: a block's slots are
    // bs / 16 consecutive groups
    cuuint64_t dims[5] = {64, 16, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(Hkv),
                          2ull * static_cast<cuuint64_t>(NB) * static_cast<cuuint64_t>(bs / 16)};
    cuuint64_t strides[4] = {row * Hkv, 128, row, 16 * row * Hkv};
    cuuint32_t box[5] = {64, 16, static_cast<cuuint32_t>(D / 64), 1,
                         static_cast<cuuint32_t>(box_rows / 16)};
    return enc(map, dt, 5, const_cast<void*>(kv_cache), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(bs), 2ull * static_cast<cuuint64_t>(NB)};
  cuuint64_t strides[3] = {row, row * Hkv, row * Hkv * bs};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  return enc(map, dt, 4, const_cast<void*>(kv_cache), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The three maps of a prefill launch: q, the K copies and the V copies.  An
// e4m3 cache's V copies (and its K copies at d 64) take the unswizzled rows.
bool encode_prefill_maps(CUtensorMap* qmap, CUtensorMap* kmap, CUtensorMap* vmap, const void* q,
                         const void* kv_cache, int kv_dtype, int H, int D, int T, int Hkv, int bs,
                         int NB) {
  const int rows = std::min(bs, BLOCK_N);
  if (!encode_q_map(qmap, q, kv_dtype, H, D, T)) return false;
  if (!encode_kv_map(kmap, kv_cache, kv_dtype, D, Hkv, bs, NB, rows, false)) return false;
  return encode_kv_map(vmap, kv_cache, kv_dtype, D, Hkv, bs, NB, rows, true);
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

bool encode_diffkv_map(CUtensorMap* map, const void* cache, int kv_dtype, int dk, int dv, int Hkv,
                       int bs, int NB, int chunks) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t row = 2ull * static_cast<cuuint64_t>(dk + dv);  // bytes of a K + V row
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(NB) * static_cast<cuuint64_t>(bs),
                        static_cast<cuuint64_t>((dk + dv) / 64), static_cast<cuuint64_t>(Hkv)};
  cuuint64_t strides[3] = {row * Hkv, 128, row};
  cuuint32_t box[4] = {64, 16, static_cast<cuuint32_t>(chunks), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map,
             kv_dtype == PATTN_KV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
             4, const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  L.order_off = off;
  off = align_up(off + static_cast<size_t>(B) * sizeof(int), 256);
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

// pattn_varlen_fwd on a DiffKV cache: the status word is cleared and the
// requests are ordered longest decode first, then the generic kernel serves
// the rows with query_len > 1 and the tensor-core DiffKV decode kernel the
// decode rows (head sizes that are multiples of 64; the generic kernel serves
// every row otherwise).
pattn_status_t diffkv_fwd(const void* q, const void* kv_cache, const int32_t* block_table,
                          const int32_t* seq_lens, const int32_t* query_start_loc, void* out,
                          float scale, int num_heads, int num_kv_heads, int head_size,
                          int block_size, int window, int causal, int kv_dtype,
                          const pattn_ext_t* ext) {
  // the standard layout with rows of the larger head size (pattn_workspace_bytes
  // sizes it the same way, for no window): header, partition counters, decode
  // order and the partitions' partial results of the tensor-core decode kernel
  const int hv = ext_head_size_v(ext);
  const int splits = diffkv_decode_supported(head_size, hv)
                         ? choose_splits(ext, num_kv_heads, block_size, window)
                         : 1;
  const WsLayout L = workspace_layout(ext->num_seqs, ext->num_tokens, num_heads, num_kv_heads,
                                      std::max(head_size, hv), ext->max_query_len, splits);
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
  p.window = window;
  p.causal = causal;
  p.kv_dtype = kv_dtype;
  p.B = ext->num_seqs;
  p.T = ext->num_tokens;
  p.mbps = ext->max_blocks_per_seq;
  p.bt_stride = p.mbps;
  p.NB = ext->num_blocks;
  p.max_q = ext->max_query_len;
  p.max_s = ext->max_seq_len;
  p.sinks = ext_sinks(ext);
  unsigned char* ws = static_cast<unsigned char*>(ext->workspace);
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.counters = reinterpret_cast<unsigned*>(ws + L.counters_off);
  p.decode_order = reinterpret_cast<int*>(ws + L.order_off);
  p.o_part = reinterpret_cast<float*>(ws + L.o_part_off);
  p.lse_part = reinterpret_cast<float*>(ws + L.lse_off);
  p.splits = splits;
  p.stream = static_cast<cudaStream_t>(ext->stream);
  // the decode kernel follows the clearing kernel as its programmatic
  // dependent (unless the caller records events between the kernels)
  p.pdl_launch = p.pdl_wait = (ext->timing_events == nullptr) ? 1 : 0;
  // clears the status word and orders the requests longest decode first (the
  // decode grid's order), then the kernels run
  if (launch_decode_prep(p) != cudaSuccess) return PATTN_ERR_CUDA;
  if (launch_diffkv(p, head_size, ext_head_size_v(ext)) != cudaSuccess) return PATTN_ERR_CUDA;
  return PATTN_OK;
}

}  // namespace pattn

using namespace pattn;

extern "C" {

int pattn_version(void) { return 10000; }

#ifdef PATTN_WAIT_TEST
void pattn_test_set_wait_skip(int mode) { g_test_wait_skip.store(mode); }
#endif

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
  // The DiffKV layout's partial rows have the larger of the two head sizes.
  const int splits = choose_splits(ext, num_kv_heads, block_size, 0);
  return workspace_layout(ext->num_seqs, ext->num_tokens, num_heads, num_kv_heads,
                          std::max(head_size, ext_head_size_v(ext)), ext->max_query_len, splits)
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
  pattn_status_t v = check_call(q, kv_cache, block_table, seq_lens, query_start_loc, out, scale,
                                num_heads, num_kv_heads, head_size, block_size, window, causal,
                                kv_dtype, kv_scale, ext);
  if (v != PATTN_OK) return v;
  if (window < 0) window = 0;
  if (ext_head_size_v(ext) > 0)
    return diffkv_fwd(q, kv_cache, block_table, seq_lens, query_start_loc, out, scale, num_heads,
                      num_kv_heads, head_size, block_size, window, causal, kv_dtype, ext);

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
  p.bt_stride = p.mbps;
  p.kv_chunks = 1;
  p.clear_status = 1;
  p.o32 = nullptr;
  p.lse32 = nullptr;
  p.sinks = ext_sinks(ext);
  p.NB = ext->num_blocks;
  p.max_q = ext->max_query_len;
  p.max_s = ext->max_seq_len;
  p.splits = splits;
  unsigned char* ws = static_cast<unsigned char*>(ext->workspace);
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.tiles = reinterpret_cast<int2*>(ws + L.tiles_off);
  p.decode_order = reinterpret_cast<int*>(ws + L.order_off);
  p.max_tiles = L.max_tiles;
  p.rows_per_item = prefill_rows_per_item(p.G);
  p.counters = reinterpret_cast<unsigned*>(ws + L.counters_off);
  p.o_part = reinterpret_cast<float*>(ws + L.o_part_off);
  p.lse_part = reinterpret_cast<float*>(ws + L.lse_off);
  p.stream = static_cast<cudaStream_t>(ext->stream);
#ifdef PATTN_WAIT_TEST
  p.test_skip = test_wait_skip();
#endif

  // Optional per-phase events (profiling): [2k] before and [2k+1] after phase k.
  auto mark = [&](int idx) {
    if (ext->timing_events && ext->timing_events[idx])
      cudaEventRecord(static_cast<cudaEvent_t>(ext->timing_events[idx]), p.stream);
  };

  // Prefill rows run on the tensor-core kernel (an e4m3 cache widened to f16
  // in its shared memory).
  const bool tc_prefill = ext->max_query_len > 1;
  // A batch with prefill rows co-schedules the two kernels (the plan kernel
  // sizes the prefill grid from the actual work; with no decode rows it keeps
  // every SM).  With per-phase events between the kernels they run one after
  // the other on every SM instead.
  p.co_schedule = (ext->timing_events == nullptr && tc_prefill) ? 1 : 0;
  set_cost_model(p);
  mark(0);
  if (tc_prefill) {
    // The plan kernel clears the header and the counters and builds the
    // prefill work list.
    if (launch_plan(p) != cudaSuccess) return PATTN_ERR_CUDA;
  } else {
    // Decode only: nothing to plan (the decode kernel validates its own
    // rows); clear the status word and the partition counters and order the
    // requests longest first.
    if (launch_decode_prep(p) != cudaSuccess) return PATTN_ERR_CUDA;
  }
  // The decode kernel is a programmatic dependent of the kernel before it,
  // unless per-phase events sit between them.  After the prep kernel it
  // waits for it before it starts (it reads the order that kernel writes);
  // after the prefill kernel (which starts only once the plan kernel's writes
  // are done) it has nothing to wait for, and it may take the SMs of finished
  // prefill CTAs.
  const bool timed = ext->timing_events != nullptr;
  p.pdl_launch = timed ? 0 : 1;
  p.pdl_wait = tc_prefill ? 0 : 1;
  p.pdl_trigger = (!timed && tc_prefill) ? 1 : 0;

  mark(1);
  mark(2);

  if (tc_prefill) {
    CUtensorMap qmap, kmap, vmap;
    if (!encode_prefill_maps(&qmap, &kmap, &vmap, q, kv_cache, kv_dtype, num_heads, head_size,
                             ext->num_tokens, num_kv_heads, block_size, ext->num_blocks))
      return PATTN_ERR_CUDA;
    if (launch_prefill(p, qmap, kmap, vmap) != cudaSuccess) return PATTN_ERR_CUDA;
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

size_t pattn_cascade_workspace_bytes(const pattn_ext_t* ext, int num_heads, int num_kv_heads,
                                     int head_size, int block_size, int common_prefix_len) {
  if (validate(ext, num_heads, num_kv_heads, head_size, block_size) != PATTN_OK) return 0;
  if (common_prefix_len <= 0 || common_prefix_len % block_size != 0) return 0;
  return cascade_layout(ext, num_heads, num_kv_heads, head_size, block_size, common_prefix_len).total;
}

pattn_status_t pattn_cascade_fwd(const void* q, const void* kv_cache, const int32_t* block_table,
                                 const int32_t* seq_lens, const int32_t* query_start_loc,
                                 void* out, float scale, int num_heads, int num_kv_heads,
                                 int head_size, int block_size, int window, int causal,
                                 int kv_dtype, const float* kv_scale, int common_prefix_len,
                                 const pattn_ext_t* ext) {
  pattn_status_t v = check_call(q, kv_cache, block_table, seq_lens, query_start_loc, out, scale,
                                num_heads, num_kv_heads, head_size, block_size, window, causal,
                                kv_dtype, kv_scale, ext);
  if (v != PATTN_OK) return v;
  if (ext_head_size_v(ext) > 0) return PATTN_ERR_UNSUPPORTED;  // DiffKV: pattn_varlen_fwd only
  const int P = common_prefix_len;
  if (P <= 0 || P % block_size != 0) return PATTN_ERR_INVALID_ARGUMENT;
  if (causal != 1 || window > 0) return PATTN_ERR_UNSUPPORTED;
  // The prefix pass is one request of every query token: its 128-key tiles
  // need the same page rule as any prefill.
  if (!(BLOCK_N % block_size == 0 || block_size % BLOCK_N == 0)) return PATTN_ERR_UNSUPPORTED;
  if (P > ext->max_seq_len || P / block_size > ext->max_blocks_per_seq)
    return PATTN_ERR_INVALID_ARGUMENT;
  const CascadeLayout c = cascade_layout(ext, num_heads, num_kv_heads, head_size, block_size, P);
  if (ext->workspace_bytes < c.total) return PATTN_ERR_WORKSPACE_TOO_SMALL;
  if (ext->num_seqs == 0 || ext->num_tokens == 0) return PATTN_OK;
  if (ext->num_blocks == 0) return PATTN_ERR_INVALID_ARGUMENT;

  unsigned char* ws = static_cast<unsigned char*>(ext->workspace);
  int* pre_qsl = reinterpret_cast<int*>(ws + c.meta);
  int* pre_sl = pre_qsl + 2;
  int* suf_sl = pre_qsl + 3;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);

  // Prefix pass: one request spanning every query token, over the first
  // P / block_size entries of block-table row 0 (the same blocks in every
  // row), not causal.  It reports into the call's status word.
  Problem pre;
  base_problem(pre, q, kv_cache, out, scale, num_heads, num_kv_heads, head_size, block_size,
               kv_dtype, kv_scale, ext);
  pre.block_table = block_table;
  pre.seq_lens = pre_sl;
  pre.qsl = pre_qsl;
  pre.window = 0;
  pre.causal = 0;
  pre.B = 1;
  pre.mbps = P / block_size;
  pre.bt_stride = ext->max_blocks_per_seq;
  pre.max_q = ext->num_tokens;
  pre.max_s = P;
  pre.splits = c.splits_pre;
  pre.hdr = hdr;
  pre.clear_status = 0;
  pre.long_queries = 1;
  pre.tiles = reinterpret_cast<int2*>(ws + c.pre_off + c.pre.tiles_off);
  pre.max_tiles = c.pre.max_tiles;
  pre.counters = reinterpret_cast<unsigned*>(ws + c.pre_off + c.pre.counters_off);
  pre.o_part = reinterpret_cast<float*>(ws + c.pre_off + c.pre.o_part_off);
  pre.lse_part = reinterpret_cast<float*>(ws + c.pre_off + c.pre.lse_off);
  pre.o32 = reinterpret_cast<float*>(ws + c.o_pre);
  pre.lse32 = reinterpret_cast<float*>(ws + c.lse_pre);
  pre.kv_chunks = (ext->num_tokens > 1) ? c.kc : 1;  // a single token runs the decode kernel

  // Suffix pass: every request over its own keys past the prefix, causal
  // (positions relative to the prefix's end), block-table rows shifted by the
  // prefix's blocks.
  Problem suf;
  base_problem(suf, q, kv_cache, out, scale, num_heads, num_kv_heads, head_size, block_size,
               kv_dtype, kv_scale, ext);
  suf.block_table = block_table + P / block_size;
  suf.seq_lens = suf_sl;
  suf.qsl = query_start_loc;
  suf.window = 0;
  suf.causal = 1;
  suf.B = ext->num_seqs;
  suf.mbps = ext->max_blocks_per_seq - P / block_size;
  suf.bt_stride = ext->max_blocks_per_seq;
  suf.max_q = ext->max_query_len;
  suf.max_s = std::max(1, ext->max_seq_len - P);
  suf.splits = c.splits_suf;
  suf.hdr = hdr;
  suf.clear_status = 0;
  suf.tiles = reinterpret_cast<int2*>(ws + c.suf.tiles_off);
  suf.max_tiles = c.suf.max_tiles;
  suf.counters = reinterpret_cast<unsigned*>(ws + c.suf.counters_off);
  suf.o_part = reinterpret_cast<float*>(ws + c.suf.o_part_off);
  suf.lse_part = reinterpret_cast<float*>(ws + c.suf.lse_off);
  suf.o32 = reinterpret_cast<float*>(ws + c.o_suf);
  suf.lse32 = reinterpret_cast<float*>(ws + c.lse_suf);

  cudaStream_t st = static_cast<cudaStream_t>(ext->stream);
  if (launch_cascade_setup(hdr, query_start_loc, seq_lens, ext->num_seqs, P, pre_qsl, pre_sl,
                           suf_sl, st) != cudaSuccess)
    return PATTN_ERR_CUDA;
  for (Problem* p : {&pre, &suf}) {
    if (p->max_q > 1) {
      if (launch_plan(*p) != cudaSuccess) return PATTN_ERR_CUDA;
    } else if (cudaMemsetAsync(p->counters, 0, static_cast<size_t>(p->B) * p->Hkv * sizeof(unsigned),
                               st) != cudaSuccess) {
      return PATTN_ERR_CUDA;
    }
    v = launch_pass(*p);
    if (v != PATTN_OK) return v;
  }
  if (launch_cascade_merge(pre.o32, pre.lse32, pre.kv_chunks, suf.o32, suf.lse32, out,
                           query_start_loc,
                           ext->num_seqs, ext->num_tokens, num_heads, head_size,
                           kv_dtype == PATTN_KV_F16, ext_sinks(ext), st) != cudaSuccess)
    return PATTN_ERR_CUDA;
  return PATTN_OK;
}

}  // extern "C"
