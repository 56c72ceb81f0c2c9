// cache_write.cu -- KV-cache write through slot_mapping (sm_103a).
//
// The step that fills the cache attention reads: FlashAttentionMetadata of
// "[vLLM] FlashAttention" carries a slot_mapping beside the block table (the
// PagedAttention point of its "why this design" list), and the DiffKV backend
// of "[vLLM] other attention backends" has its own cache-write kernel for its
// asymmetric cache shape.  Token t with slot s = slot_mapping[t] >= 0 writes
// its key and value rows of every KV head to cache[0 or 1][s / bs][s % bs];
// a negative slot writes nothing.  For an e4m3 cache each element is stored
// as e4m3(x / scale) of the fp32 quotient (IEEE division), rounded to nearest
// even and saturated at +-448 by CUDA's conversion intrinsic.
//
// Pure data movement, bound by HBM: each thread moves 16 bytes of one key or
// value row (8 bf16 elements), so a warp covers two 256-byte rows (head size
// 128) with fully coalesced loads and stores.
#include "../../include/pattn.h"
#include "common.cuh"

namespace pattn {
namespace {

constexpr int CW_THREADS = 256;

template <bool FP8>
__global__ void __launch_bounds__(CW_THREADS)
    reshape_and_cache_kernel(const __nv_bfloat16* __restrict__ key,
                             const __nv_bfloat16* __restrict__ value, void* __restrict__ cache,
                             const int64_t* __restrict__ slots, int T, int Hkv, int D, int bs,
                             int NB, float k_scale, float v_scale, unsigned* status) {
  const int chunks = D / 8;                            // 16-byte pieces of a row
  const int64_t per_token = 2LL * Hkv * chunks;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * CW_THREADS + threadIdx.x;
  if (idx >= per_token * T) return;
  const int t = static_cast<int>(idx / per_token);
  int rem = static_cast<int>(idx - static_cast<int64_t>(t) * per_token);
  const int kv = rem / (Hkv * chunks);
  rem -= kv * Hkv * chunks;
  const int h = rem / chunks, c = rem - h * chunks;
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= static_cast<int64_t>(NB) * bs) {
    if (kv == 0 && h == 0 && c == 0 && status) atomicOr(status, PATTN_DEV_BAD_METADATA);
    return;
  }
  const int64_t blk = s / bs, off = s - blk * bs;
  const __nv_bfloat16* src = (kv ? value : key) + (static_cast<int64_t>(t) * Hkv + h) * D + c * 8;
  const int64_t dst = ((((kv * static_cast<int64_t>(NB) + blk) * bs + off) * Hkv + h) * D) + c * 8;
  const uint4 x = *reinterpret_cast<const uint4*>(src);
  if constexpr (!FP8) {
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(cache) + dst) = x;
  } else {
    const float sc = kv ? v_scale : k_scale;
    const unsigned w[4] = {x.x, x.y, x.z, x.w};
    unsigned packed[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const unsigned short bits = static_cast<unsigned short>(w[e >> 1] >> ((e & 1) * 16));
      const float v = __bfloat162float(__ushort_as_bfloat16(bits));
      const __nv_fp8_storage_t b = __nv_cvt_float_to_fp8(__fdiv_rn(v, sc), __NV_SATFINITE, __NV_E4M3);
      packed[e >> 2] |= static_cast<unsigned>(b) << ((e & 3) * 8);
    }
    *reinterpret_cast<uint2*>(static_cast<unsigned char*>(cache) + dst) = make_uint2(packed[0], packed[1]);
  }
}

// DiffKV layout [NB][bs][Hkv][dk + dv]: token t's key row (dk elements) then
// its value row (dv) go to cache row [s / bs][s % bs][h].  16-bit data only;
// each thread moves 16 bytes (8 elements) of one key or value row.
__global__ void __launch_bounds__(CW_THREADS)
    reshape_and_cache_diffkv_kernel(const uint16_t* __restrict__ key,
                                    const uint16_t* __restrict__ value, uint16_t* __restrict__ cache,
                                    const int64_t* __restrict__ slots, int T, int Hkv, int dk,
                                    int dv, int bs, int NB, unsigned* status) {
  const int ck = dk / 8, cv = dv / 8;                  // 16-byte pieces of a K / V row
  const int64_t per_token = static_cast<int64_t>(Hkv) * (ck + cv);
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * CW_THREADS + threadIdx.x;
  if (idx >= per_token * T) return;
  const int t = static_cast<int>(idx / per_token);
  const int rem = static_cast<int>(idx - static_cast<int64_t>(t) * per_token);
  const int h = rem / (ck + cv), c = rem - h * (ck + cv);
  const int64_t s = slots[t];
  if (s < 0) return;
  if (s >= static_cast<int64_t>(NB) * bs) {
    if (h == 0 && c == 0 && status) atomicOr(status, PATTN_DEV_BAD_METADATA);
    return;
  }
  const bool is_v = c >= ck;
  const uint16_t* src = is_v ? value + (static_cast<int64_t>(t) * Hkv + h) * dv + (c - ck) * 8
                             : key + (static_cast<int64_t>(t) * Hkv + h) * dk + c * 8;
  const int64_t dst = (s * Hkv + h) * static_cast<int64_t>(dk + dv) + c * 8;
  *reinterpret_cast<uint4*>(cache + dst) = *reinterpret_cast<const uint4*>(src);
}

}  // namespace
}  // namespace pattn

using namespace pattn;

extern "C" pattn_status_t pattn_reshape_and_cache_diffkv(
    const void* key, const void* value, void* kv_cache, const int64_t* slot_mapping,
    int num_tokens, int num_kv_heads, int head_size, int head_size_v, int block_size,
    int num_blocks, int kv_dtype, unsigned* device_status, void* stream) {
  if (!key || !value || !kv_cache || !slot_mapping) return PATTN_ERR_INVALID_ARGUMENT;
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks < 0) return PATTN_ERR_INVALID_ARGUMENT;
  if (block_size <= 0 || block_size % 16 != 0) return PATTN_ERR_INVALID_ARGUMENT;
  if (head_size <= 0 || head_size % 8 != 0 || head_size_v <= 0 || head_size_v % 8 != 0)
    return PATTN_ERR_UNSUPPORTED;
  if (kv_dtype != PATTN_KV_BF16 && kv_dtype != PATTN_KV_F16) return PATTN_ERR_UNSUPPORTED;
  const uintptr_t align = reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value) |
                          reinterpret_cast<uintptr_t>(kv_cache);
  if (align & 15) return PATTN_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return PATTN_OK;
  const long long n =
      static_cast<long long>(num_tokens) * num_kv_heads * ((head_size + head_size_v) / 8);
  const unsigned grid = static_cast<unsigned>((n + CW_THREADS - 1) / CW_THREADS);
  reshape_and_cache_diffkv_kernel<<<grid, CW_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(key), static_cast<const uint16_t*>(value),
      static_cast<uint16_t*>(kv_cache), slot_mapping, num_tokens, num_kv_heads, head_size,
      head_size_v, block_size, num_blocks, device_status);
  return cudaGetLastError() == cudaSuccess ? PATTN_OK : PATTN_ERR_CUDA;
}

extern "C" pattn_status_t pattn_reshape_and_cache(const void* key, const void* value,
                                                  void* kv_cache, const int64_t* slot_mapping,
                                                  int num_tokens, int num_kv_heads, int head_size,
                                                  int block_size, int num_blocks, int kv_dtype,
                                                  const float* kv_scale, unsigned* device_status,
                                                  void* stream) {
  if (!key || !value || !kv_cache || !slot_mapping) return PATTN_ERR_INVALID_ARGUMENT;
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks < 0) return PATTN_ERR_INVALID_ARGUMENT;
  if (block_size <= 0 || block_size % 16 != 0) return PATTN_ERR_INVALID_ARGUMENT;
  if (head_size <= 0 || head_size % 8 != 0) return PATTN_ERR_UNSUPPORTED;
  if (kv_dtype != PATTN_KV_BF16 && kv_dtype != PATTN_KV_FP8_E4M3 && kv_dtype != PATTN_KV_F16)
    return PATTN_ERR_UNSUPPORTED;
  if (kv_dtype == PATTN_KV_FP8_E4M3 &&
      (!kv_scale || !(kv_scale[0] > 0.f) || !(kv_scale[1] > 0.f) || !(kv_scale[0] < INFINITY) ||
       !(kv_scale[1] < INFINITY)))
    return PATTN_ERR_INVALID_ARGUMENT;
  const uintptr_t align = reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value) |
                          reinterpret_cast<uintptr_t>(kv_cache);
  if (align & 15) return PATTN_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return PATTN_OK;
  const long long n = static_cast<long long>(num_tokens) * 2 * num_kv_heads * (head_size / 8);
  const unsigned grid = static_cast<unsigned>((n + CW_THREADS - 1) / CW_THREADS);
  const bool fp8 = kv_dtype == PATTN_KV_FP8_E4M3;
  const float ks = fp8 ? kv_scale[0] : 1.f, vs = fp8 ? kv_scale[1] : 1.f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const auto* k = static_cast<const __nv_bfloat16*>(key);
  const auto* v = static_cast<const __nv_bfloat16*>(value);
  if (kv_dtype == PATTN_KV_FP8_E4M3)
    reshape_and_cache_kernel<true><<<grid, CW_THREADS, 0, st>>>(
        k, v, kv_cache, slot_mapping, num_tokens, num_kv_heads, head_size, block_size, num_blocks,
        ks, vs, device_status);
  else
    reshape_and_cache_kernel<false><<<grid, CW_THREADS, 0, st>>>(
        k, v, kv_cache, slot_mapping, num_tokens, num_kv_heads, head_size, block_size, num_blocks,
        ks, vs, device_status);
  return cudaGetLastError() == cudaSuccess ? PATTN_OK : PATTN_ERR_CUDA;
}
