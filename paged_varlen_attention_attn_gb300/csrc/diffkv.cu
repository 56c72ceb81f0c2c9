// diffkv.cu -- attention over a DiffKV cache, where V has its own head size
// (sm_103a).
//
// "[vLLM] other attention backends", FlashAttention DiffKV: the head size of V
// (head_size_v) may differ from that of K, and the KV cache is then
// asymmetric.  The page gives no shape; the layout read here is one tensor
// [num_blocks][block_size][num_kv_heads][dk + dv], each row holding the
// token's K (dk elements) and then its V (dv elements).  The attention is
// pattn_varlen_fwd's (causal or not, sliding window, GQA, sinks); out is
// [T][H][dv].
//
// This generic SIMT kernel serves the rows with query_len > 1 (the decode
// rows run on the tensor-core kernel of diffkv_decode.cu when dk and dv are
// multiples of 64; otherwise this kernel serves them too), for any dk, dv that
// are multiples of 32 up to 256.  One CTA per (query token, KV head): its four warps
// share the KV head's G query heads (warp w takes heads w, w + 4, ...).  Key
// tiles of 32 rows (K and V together) are copied into shared memory with
// 16-byte cp.async (rows past the visible range zero-filled), double
// buffered so the next tile streams in while the current one is used.  Each
// staged row is padded by 16 bytes, so the 16-byte reads of lane k in row k
// fall on distinct banks within every quarter warp.  Lane k scores key k of
// the tile; the online softmax runs in log2 units; lane j accumulates output
// columns j, j + 32, ... of each of its heads.
#include "../../include/pattn.h"
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

constexpr int DKV_THREADS = 128;
constexpr int DKV_KEYS = 32;   // keys per staged tile
constexpr int DKV_MAXH = 4;    // query heads per warp: G <= 16
constexpr unsigned FULL_MASK = 0xffffffffu;

template <bool HALF>
__device__ __forceinline__ float2 unpack2(unsigned w) {
  if constexpr (HALF) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  } else {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
}

template <bool HALF>
__device__ __forceinline__ float elem(const void* base, int64_t i) {
  if constexpr (HALF)
    return __half2float(static_cast<const __half*>(base)[i]);
  else
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
}

template <bool HALF>
__device__ __forceinline__ void store(void* base, int64_t i, float v) {
  if constexpr (HALF)
    static_cast<__half*>(base)[i] = __float2half_rn(v);
  else
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL_MASK, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src, bool valid) {
  // src-size 0 fills the 16 bytes with zeros and reads nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool HALF>
__device__ __forceinline__ float half_bits_to_float(unsigned short b) {
  if constexpr (HALF)
    return __half2float(__ushort_as_half(b));
  else
    return __bfloat162float(__ushort_as_bfloat16(b));
}

// (d0, d1) += (a0, a1) * (b0, b1) on the paired fp32 pipe
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rd, {%0, %1};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rd;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// dot(q[0..7], 8 16-bit values in w) into (d0, d1)
template <bool HALF>
__device__ __forceinline__ void dot8(const float4 qa, const float4 qb, const uint4 w, float& d0,
                                     float& d1) {
  float2 f = unpack2<HALF>(w.x);
  fma2(d0, d1, qa.x, qa.y, f.x, f.y);
  f = unpack2<HALF>(w.y);
  fma2(d0, d1, qa.z, qa.w, f.x, f.y);
  f = unpack2<HALF>(w.z);
  fma2(d0, d1, qb.x, qb.y, f.x, f.y);
  f = unpack2<HALF>(w.w);
  fma2(d0, d1, qb.z, qb.w, f.x, f.y);
}

// HALF: q, the cache and out are f16 (else bf16).
// NC: dv / 32, the output columns per lane.  With NC even a lane owns pairs of
// adjacent columns (2 lane + 64 c, + 1), read as one 32-bit word per key and
// stored together; with NC odd, columns lane + 32 c.
// skip_decode: rows of requests with query_len 1 are left to the decode kernel.
template <bool HALF, int NC>
__global__ void __launch_bounds__(DKV_THREADS)
    diffkv_kernel(const __grid_constant__ Problem p, int dk, int dv, float sl2, int skip_decode) {
  constexpr int ES = 2;
  extern __shared__ __align__(16) unsigned char smem[];
  const int kbytes = dk * ES;
  const int rbytes = (dk + dv) * ES;  // a staged row: K then V
  const int rs = rbytes + 16;         // staged row stride
  const int cpr = rbytes / 16;        // 16-byte pieces of a row
  const int ck = kbytes / 16;         // ... of its K part
  float* q_s = reinterpret_cast<float*>(smem + 2 * DKV_KEYS * rs);   // [G][dk]
  const int t = blockIdx.x, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  unsigned* status = &p.hdr->status;

  // The request holding token t: the largest r with qsl[r] <= t.
  if (t < p.qsl[0] || t >= p.qsl[p.B]) return;
  int rl = 0, rh = p.B - 1;
  while (rl < rh) {
    const int mid = (rl + rh + 1) >> 1;
    if (p.qsl[mid] <= t) rl = mid;
    else rh = mid - 1;
  }
  const int r = rl;
  const int t0 = p.qsl[r], q_len = p.qsl[r + 1] - t0, s = p.seq_lens[r];
  if (skip_decode && q_len == 1) return;
  const int64_t orow = (static_cast<int64_t>(t) * p.H + static_cast<int64_t>(g) * G) * dv;
  if (t >= t0 + q_len || q_len > s || s > p.mbps * p.bs) {
    // bad metadata: reported, the row's heads written as zeros
    if (threadIdx.x == 0) flag_status(status, PATTN_DEV_BAD_METADATA);
    for (int e = threadIdx.x; e < G * dv; e += DKV_THREADS) store<HALF>(p.out, orow + e, 0.f);
    return;
  }
  const int pos = s - q_len + (t - t0);
  const int hi = p.causal ? pos + 1 : s;
  const int lo = (p.window > 0) ? max(0, pos - p.window + 1) : 0;
  const int* bt = p.block_table + static_cast<int64_t>(r) * p.bt_stride;
  const unsigned char* cache = static_cast<const unsigned char*>(p.kv);
  // bytes of a cache row (K then V)
  const int64_t src_row = rbytes;

  // Copy keys k0 .. k0 + 31 into buffer b: warp w copies rows w, w + 4, ...
  // The 32 keys' row offsets come from one coalesced block-table load (lane
  // = key) and reach each row's copy through a shuffle.
  auto stage = [&](int b, int k0) {
    unsigned char* dst = smem + b * DKV_KEYS * rs;
    const int kl = k0 + lane;
    int64_t row_off = -1;  // byte offset of key kl's row, or -1 past the range
    if (kl < hi) {
      int blk = bt[kl / p.bs];
      if (blk < 0 || blk >= p.NB) {
        flag_status(status, PATTN_DEV_BAD_METADATA);
        blk = min(max(blk, 0), p.NB - 1);
      }
      row_off = ((static_cast<int64_t>(blk) * p.bs + kl % p.bs) * p.Hkv + g) * src_row;
    }
#pragma unroll
    for (int kk = warp; kk < DKV_KEYS; kk += 4) {
      const int64_t off = __shfl_sync(FULL_MASK, row_off, kk);
      const bool ok = off >= 0;
      const unsigned char* src = cache + (ok ? off : 0);
      for (int c = lane; c < cpr; c += 32)
        cp_async16(dst + kk * rs + c * 16, src + (ok ? c * 16 : 0), ok);
    }
    cp_async_commit();
  };

  const int ntiles = (hi > lo) ? (hi - lo + DKV_KEYS - 1) / DKV_KEYS : 0;
  if (ntiles > 0) stage(0, lo);

  // q of the G heads, as floats
  const int64_t qrow = (static_cast<int64_t>(t) * p.H + static_cast<int64_t>(g) * G) * dk;
  for (int e = threadIdx.x; e < G * dk; e += DKV_THREADS) q_s[e] = elem<HALF>(p.q, qrow + e);

  constexpr bool PAIRS = (NC % 2) == 0;
  float m_run[DKV_MAXH], l_run[DKV_MAXH], o[DKV_MAXH][NC];
#pragma unroll
  for (int jh = 0; jh < DKV_MAXH; ++jh) {
    m_run[jh] = -INFINITY;
    l_run[jh] = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) o[jh][c] = 0.f;
  }

  for (int j = 0; j < ntiles; ++j) {
    const int k0 = lo + j * DKV_KEYS;
    if (j + 1 < ntiles) {
      stage((j + 1) & 1, k0 + DKV_KEYS);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // tile j (and q) in shared memory for every thread
    const unsigned char* tb = smem + (j & 1) * DKV_KEYS * rs;
    const bool key_ok = k0 + lane < hi;
#pragma unroll
    for (int jh = 0; jh < DKV_MAXH; ++jh) {
      const int hh = warp + 4 * jh;  // query head within the group
      if (hh >= G) continue;
      // score of key k0 + lane
      const float4* q4 = reinterpret_cast<const float4*>(q_s + hh * dk);
      const uint4* krow = reinterpret_cast<const uint4*>(tb + lane * rs);
      float dot0 = 0.f, dot1 = 0.f;
#pragma unroll 4
      for (int c = 0; c < ck; ++c) {
        dot8<HALF>(q4[2 * c], q4[2 * c + 1], krow[c], dot0, dot1);  // 8 16-bit values
      }
      const float s2 = key_ok ? (dot0 + dot1) * sl2 : -INFINITY;
      const float m_new = fmaxf(m_run[jh], warp_max(s2));
      if (m_new == -INFINITY) continue;  // nothing visible yet
      const float alpha = fast_exp2(m_run[jh] - m_new);
      const float pk = fast_exp2(s2 - m_new);
      l_run[jh] = l_run[jh] * alpha + warp_sum(pk);
      m_run[jh] = m_new;
#pragma unroll
      for (int c = 0; c < NC; ++c) o[jh][c] *= alpha;
      // o += sum_k p_k V_k over this lane's columns
#pragma unroll 8
      for (int kk = 0; kk < DKV_KEYS; ++kk) {
        const float pb = __shfl_sync(FULL_MASK, pk, kk);
        const unsigned char* vbase = tb + kk * rs + kbytes;
        if constexpr (PAIRS) {
#pragma unroll
          for (int c2 = 0; c2 < NC / 2; ++c2) {
            const float2 v = unpack2<HALF>(reinterpret_cast<const unsigned*>(vbase)[lane + 32 * c2]);
            fma2(o[jh][2 * c2], o[jh][2 * c2 + 1], pb, pb, v.x, v.y);
          }
        } else {
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const float v =
                half_bits_to_float<HALF>(reinterpret_cast<const unsigned short*>(vbase)[lane + 32 * c]);
            o[jh][c] = fmaf(pb, v, o[jh][c]);
          }
        }
      }
    }
    __syncthreads();  // tile j used: its buffer may be refilled
  }

  // normalise (with the head's sink) and write
#pragma unroll
  for (int jh = 0; jh < DKV_MAXH; ++jh) {
    const int hh = warp + 4 * jh;
    if (hh >= G) continue;
    const float l_tot = l_run[jh] + sink_term(p.sinks, g * G + hh, m_run[jh]);
    const float inv = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
    const int64_t ob = orow + static_cast<int64_t>(hh) * dv;
    if constexpr (PAIRS) {
#pragma unroll
      for (int c2 = 0; c2 < NC / 2; ++c2)
        reinterpret_cast<unsigned*>(p.out)[(ob >> 1) + lane + 32 * c2] =
            pack2<HALF>(o[jh][2 * c2] * inv, o[jh][2 * c2 + 1] * inv);
    } else {
#pragma unroll
      for (int c = 0; c < NC; ++c) store<HALF>(p.out, ob + lane + 32 * c, o[jh][c] * inv);
    }
  }
}

}  // namespace

size_t generic_smem_bytes(int G, int dk, int dv) {
  return 2 * static_cast<size_t>(DKV_KEYS) * ((dk + dv) * 2 + 16) +
         static_cast<size_t>(G) * dk * sizeof(float);
}

template <bool HALF, int NC>
cudaError_t launch_generic_t(const Problem& p, int dk, int dv, bool skip_decode) {
  const size_t smem = generic_smem_bytes(p.G, dk, dv);
  const float sl2 = fmaxf(p.scale * LOG2E, 1e-30f);
  const dim3 grid(static_cast<unsigned>(p.T), static_cast<unsigned>(p.Hkv));
  auto kern = diffkv_kernel<HALF, NC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, DKV_THREADS, smem, p.stream>>>(p, dk, dv, sl2, skip_decode ? 1 : 0);
  return cudaGetLastError();
}

template <bool HALF>
cudaError_t launch_generic_h(const Problem& p, int dk, int dv, bool skip_decode) {
  switch (dv / 32) {
    case 1: return launch_generic_t<HALF, 1>(p, dk, dv, skip_decode);
    case 2: return launch_generic_t<HALF, 2>(p, dk, dv, skip_decode);
    case 3: return launch_generic_t<HALF, 3>(p, dk, dv, skip_decode);
    case 4: return launch_generic_t<HALF, 4>(p, dk, dv, skip_decode);
    case 5: return launch_generic_t<HALF, 5>(p, dk, dv, skip_decode);
    case 6: return launch_generic_t<HALF, 6>(p, dk, dv, skip_decode);
    case 7: return launch_generic_t<HALF, 7>(p, dk, dv, skip_decode);
    case 8: return launch_generic_t<HALF, 8>(p, dk, dv, skip_decode);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_generic(const Problem& p, int dk, int dv, bool skip_decode) {
  if (p.T == 0 || p.B == 0) return cudaSuccess;
  return p.kv_dtype == PATTN_KV_F16 ? launch_generic_h<true>(p, dk, dv, skip_decode)
                                    : launch_generic_h<false>(p, dk, dv, skip_decode);
}

// Rows with query_len > 1 on the generic kernel (when the batch may have
// them), then the decode rows on the tensor-core kernel; head sizes that are
// not multiples of 64 run every row on the generic kernel.
// The decode kernel is the clearing kernel's programmatic dependent only when
// it follows that kernel directly (p.pdl_launch / pdl_wait from the caller).
cudaError_t launch_diffkv(const Problem& p, int dk, int dv) {
  if (!diffkv_decode_supported(dk, dv)) return launch_generic(p, dk, dv, false);
  if (p.max_q > 1) {
    const cudaError_t e = launch_generic(p, dk, dv, true);
    if (e != cudaSuccess) return e;
    Problem after = p;
    after.pdl_launch = after.pdl_wait = 0;
    return launch_diffkv_decode(after, dk, dv);
  }
  return launch_diffkv_decode(p, dk, dv);
}

}  // namespace pattn
