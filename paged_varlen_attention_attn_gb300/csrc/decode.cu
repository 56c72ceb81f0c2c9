// decode.cu -- split-KV decode kernel and log-sum-exp combine (sm_103a).
//
// Decode rows (query_len == 1; the prefill/decode split with threshold 1 of
// "[vLLM] Lightning & Linear Attention") are bound by reading K/V from HBM:
// each KV byte feeds 2G (bf16) FLOPs, far below the tensor ridge.  One CTA
// takes one (request, KV head, partition) item, so the G query heads of a KV
// head share every page it reads (FlashAttentionImpl's num_queries_per_kv).
// The partition is a run of whole KV blocks ("RBLN Attention modes": flash
// attention processes the cache by partitions and merges them with online
// softmax); partial results go to the workspace as (o_p, lse_p) and
// combine_kernel merges them, or the CTA writes the output directly when
// there is one partition.
//
// Data path: each warp streams 16-key units (one unit never straddles a KV
// block because block_size % 16 == 0) through its own cp.async ring of
// 16-byte vectors, with a 128-byte XOR swizzle so ldmatrix reads are
// conflict-free.  Scores and P.V run on mma.sync m16n8k16 with the G heads as
// the M rows: at G <= 8 that wastes half the MMA rows, which costs nothing
// here because the kernel waits on HBM.  e4m3 units are widened to f16 in
// shared memory (exact: every e4m3 value is an f16 value) by CUDA's paired
// conversion intrinsic; the per-tensor scales are folded into the softmax
// scale (K) and the final normalisation (V).
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

constexpr int DEC_WARPS = 4;
constexpr int DEC_STAGES = 3;
constexpr int UNIT = 16;  // keys per unit

template <int D, bool FP8>
struct DecodeCfg {
  static constexpr int ES = FP8 ? 1 : 2;
  static constexpr int RAW_ROW = D * ES;            // bytes of one key row in the cache
  static constexpr int RAW_UNIT = UNIT * RAW_ROW;   // bytes of one K (or V) unit
  static constexpr int H_ROW = D * 2;               // 16-bit row in shared memory
  static constexpr int H_UNIT = UNIT * H_ROW;
  static constexpr int STAGE = 2 * RAW_UNIT;        // K + V raw unit
  // per warp: stages + (fp8 only) one widened K/V unit pair
  static constexpr int WARP_BYTES = DEC_STAGES * STAGE + (FP8 ? 2 * H_UNIT : 0);
  static constexpr int SMEM = DEC_WARPS * WARP_BYTES;
  static constexpr int MERGE_BYTES = DEC_WARPS * (16 * D + 32) * 4;
  static constexpr int SMEM_TOTAL = SMEM > MERGE_BYTES ? SMEM : MERGE_BYTES;
};

// Byte offset of 16-byte chunk c of row j in a swizzled 16-bit unit.
template <int D>
__device__ __forceinline__ int swz(int j, int c) {
  return j * (D * 2) + ((c ^ (j & 7)) << 4);
}

template <int D, bool FP8>
__global__ void __launch_bounds__(DEC_WARPS * 32)
    decode_split_kernel(const Problem p, float sl2, float out_scale) {
  using C = DecodeCfg<D, FP8>;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int S = p.splits;
  const int item = blockIdx.x;
  const int sp = item % S;
  const int g = (item / S) % p.Hkv;
  const int r = item / (S * p.Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;

  const int t0 = p.qsl[r];
  const int q_len = p.qsl[r + 1] - t0;
  if (q_len != 1) return;
  int s = p.seq_lens[r];
  bool bad = (s < 1) || (s > p.mbps * p.bs) || (t0 < 0) || (t0 >= p.T);
  unsigned* status = &p.hdr->status;
  if (bad) {
    if (threadIdx.x == 0 && sp == 0) flag_status(status, PATTN_DEV_BAD_METADATA);
    if (t0 < 0 || t0 >= p.T) return;
    s = 0;  // treat as empty: the rows become zero
  }

  // Visible keys of the decode row (p = s - 1): [k_lo, s).
  const int k_lo = (p.window > 0) ? max(0, s - p.window) : 0;
  const int b_lo = k_lo / p.bs, b_hi = (s + p.bs - 1) / p.bs;
  const int nblk = max(0, b_hi - b_lo);
  const int per = (nblk + S - 1) / S;
  const int kb = max(k_lo, (b_lo + sp * per) * p.bs);
  const int ke = min(s, (b_lo + (sp + 1) * per) * p.bs);

  const int* bt = p.block_table + static_cast<int64_t>(r) * p.mbps;
  const unsigned char* kvb = static_cast<const unsigned char*>(p.kv);
  const int64_t row_stride = static_cast<int64_t>(p.Hkv) * C::RAW_ROW;          // bytes per slot
  const int64_t v_plane = static_cast<int64_t>(p.NB) * p.bs * row_stride;        // K -> V

  // ---------------------------------------------------------------- Q in registers
  // A fragments of m16n8k16: rows = heads of this KV group (zero past G).
  unsigned qa[D / 16][4];
  {
    const int rA = lane >> 2, c2 = (lane & 3) * 2;
    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                (static_cast<int64_t>(t0) * p.H + g * G) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = rA + ((e & 1) ? 8 : 0);
        const int col = kk * 16 + c2 + ((e & 2) ? 8 : 0);
        unsigned v = 0;
        if (row < G) {
          __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(qrow + row * D + col);
          if constexpr (FP8) {
            float2 f = __bfloat1622float2(x);
            v = pack2<true>(f.x, f.y);
          } else {
            v = *reinterpret_cast<unsigned*>(&x);
          }
        }
        qa[kk][e] = v;
      }
    }
  }

  // ---------------------------------------------------------------- stream units
  const int u_begin = kb / UNIT;
  const int u_end = (ke + UNIT - 1) / UNIT;
  const int n_units = (ke > kb) ? (u_end - u_begin) : 0;
  const int my_units = (n_units > warp) ? (n_units - warp + DEC_WARPS - 1) / DEC_WARPS : 0;

  unsigned char* wbase = smem + warp * C::WARP_BYTES;
  auto stage_ptr = [&](int st) { return wbase + st * C::STAGE; };

  // Issue the loads of this warp's i-th unit into stage st.  Rows whose key
  // is at or past seq_len are written as zeros instead (their slots may hold
  // anything, NaN included).
  auto issue = [&](int i, int st) {
    const int u = u_begin + warp + i * DEC_WARPS;
    const int key0 = u * UNIT;
    int blk = bt[key0 / p.bs];
    if (blk < 0 || blk >= p.NB) {
      flag_status(status, PATTN_DEV_BAD_METADATA);
      blk = min(max(blk, 0), p.NB - 1);
    }
    const unsigned char* ksrc =
        kvb + (static_cast<int64_t>(blk) * p.bs + (key0 % p.bs)) * row_stride +
        static_cast<int64_t>(g) * C::RAW_ROW;
    unsigned char* dk = stage_ptr(st);
    unsigned char* dv = dk + C::RAW_UNIT;
    constexpr int CH_ROW = C::RAW_ROW / 16;   // 16-byte chunks per row
    constexpr int CH = UNIT * CH_ROW;          // per K (or V) unit
#pragma unroll
    for (int c = lane; c < CH; c += 32) {
      const int j = c / CH_ROW, cc = c % CH_ROW;
      // bf16 rows are stored swizzled for ldmatrix; e4m3 rows stay linear
      // (they are widened into a swizzled buffer before use).
      const int off = FP8 ? (j * C::RAW_ROW + cc * 16) : swz<D>(j, cc);
      if (key0 + j < s) {
        const unsigned char* src = ksrc + j * row_stride + cc * 16;
        cp_async_16(dk + off, src);
        cp_async_16(dv + off, src + v_plane);
      } else {
        *reinterpret_cast<uint4*>(dk + off) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(dv + off) = make_uint4(0, 0, 0, 0);
      }
    }
  };

#pragma unroll
  for (int i = 0; i < DEC_STAGES - 1; ++i) {
    if (i < my_units) issue(i, i);
    cp_async_commit();
  }

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  const int kmin = kb, kmax = ke;

  for (int i = 0; i < my_units; ++i) {
    if (i + DEC_STAGES - 1 < my_units) issue(i + DEC_STAGES - 1, (i + DEC_STAGES - 1) % DEC_STAGES);
    cp_async_commit();
    cp_async_wait<DEC_STAGES - 1>();
    __syncwarp();

    unsigned char* sk = stage_ptr(i % DEC_STAGES);
    unsigned char* sv = sk + C::RAW_UNIT;
    if constexpr (FP8) {
      // widen e4m3 -> f16 into the swizzled 16-bit buffers
      unsigned char* hk = wbase + DEC_STAGES * C::STAGE;
      unsigned char* hv = hk + C::H_UNIT;
      constexpr int CH_ROW = C::RAW_ROW / 16;
#pragma unroll
      for (int c = lane; c < UNIT * CH_ROW; c += 32) {
        const int j = c / CH_ROW, cc = c % CH_ROW;
#pragma unroll
        for (int kvi = 0; kvi < 2; ++kvi) {
          const uint4 raw = *reinterpret_cast<const uint4*>((kvi ? sv : sk) + j * C::RAW_ROW + cc * 16);
          const unsigned w[4] = {raw.x, raw.y, raw.z, raw.w};
          unsigned h[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>(w[q] & 0xFFFF), __NV_E4M3);
            __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>(w[q] >> 16), __NV_E4M3);
            h[2 * q] = *reinterpret_cast<unsigned*>(&lo);
            h[2 * q + 1] = *reinterpret_cast<unsigned*>(&hi);
          }
          unsigned char* dst = kvi ? hv : hk;
          *reinterpret_cast<uint4*>(dst + swz<D>(j, 2 * cc)) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4*>(dst + swz<D>(j, 2 * cc + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
      }
      __syncwarp();
      sk = hk;
      sv = hv;
    }

    // S = Q K^T for the 16 keys of this unit (two n8 tiles).
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const unsigned sk_a = smem_u32(sk), sv_a = smem_u32(sv);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int row = (lane & 7) + ((lane >> 4) << 3);
      const int chunk = 2 * kk + ((lane >> 3) & 1);
      unsigned b00, b01, b10, b11;
      ldsm_x4(sk_a + swz<D>(row, chunk), b00, b01, b10, b11);
      mma_16816<FP8>(sc[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b00, b01);
      mma_16816<FP8>(sc[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b10, b11);
    }

    // Mask, scale to log2 units, online softmax.
    const int u = u_begin + warp + i * DEC_WARPS;
    const int kbase = u * UNIT + (lane & 3) * 2;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = kbase + n * 8 + (e & 1);
        const float x = (k >= kmin && k < kmax) ? sc[n][e] * sl2 : -INFINITY;
        sc[n][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    float alpha[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
      const float m_new = fmaxf(m_run[hr], mx[hr]);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[hr] = fast_exp2(m_run[hr] - m_use);
      m_run[hr] = m_new;
      mx[hr] = m_use;
    }
    float ps[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = fast_exp2(sc[n][e] - mx[e >> 1]);
        sc[n][e] = pv;
        ps[e >> 1] += pv;
      }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) l_run[hr] = l_run[hr] * alpha[hr] + ps[hr];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    const unsigned pa0 = pack2<FP8>(sc[0][0], sc[0][1]);
    const unsigned pa1 = pack2<FP8>(sc[0][2], sc[0][3]);
    const unsigned pa2 = pack2<FP8>(sc[1][0], sc[1][1]);
    const unsigned pa3 = pack2<FP8>(sc[1][2], sc[1][3]);

    // O += P V: V rows are keys; ldmatrix.trans yields the col-major B fragments.
#pragma unroll
    for (int nd = 0; nd < D / 16; ++nd) {
      const int row = (lane & 7) + (((lane >> 3) & 1) << 3);
      const int chunk = 2 * nd + (lane >> 4);
      unsigned v0, v1, v2, v3;
      ldsm_x4_t(sv_a + swz<D>(row, chunk), v0, v1, v2, v3);
      mma_16816<FP8>(o[2 * nd], pa0, pa1, pa2, pa3, v0, v1);
      mma_16816<FP8>(o[2 * nd + 1], pa0, pa1, pa2, pa3, v2, v3);
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // Row sums were per lane: finish them across the quad.
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
    l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
  }

  // ---------------------------------------------------------------- merge warps
  __syncthreads();
  float* mo = reinterpret_cast<float*>(smem);                // [WARPS][16][D]
  float* mm = mo + DEC_WARPS * 16 * D;                       // [WARPS][16]
  float* ml = mm + DEC_WARPS * 16;                           // [WARPS][16]
  {
    const int rA = lane >> 2, c2 = (lane & 3) * 2;
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = rA + ((e & 2) ? 8 : 0);
        mo[(warp * 16 + row) * D + n * 8 + c2 + (e & 1)] = o[n][e];
      }
    if ((lane & 3) == 0) {
      mm[warp * 16 + rA] = m_run[0];
      mm[warp * 16 + rA + 8] = m_run[1];
      ml[warp * 16 + rA] = l_run[0];
      ml[warp * 16 + rA + 8] = l_run[1];
    }
  }
  __syncthreads();

  const int h0 = g * G;
  for (int idx = threadIdx.x; idx < G * D; idx += DEC_WARPS * 32) {
    const int row = idx / D, col = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, mm[w * 16 + row]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) {
      const float wt = fast_exp2(mm[w * 16 + row] - Mu);
      L += wt * ml[w * 16 + row];
      acc += wt * mo[(w * 16 + row) * D + col];
    }
    const float val = (L > 0.f) ? acc / L * out_scale : 0.f;
    if (S == 1) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
      out[(static_cast<int64_t>(t0) * p.H + h0 + row) * D + col] = __float2bfloat16_rn(val);
    } else {
      const int64_t prow = (static_cast<int64_t>(r) * p.H + h0 + row) * S + sp;
      p.o_part[prow * D + col] = val;
      if (col == 0) p.lse_part[prow] = (L > 0.f) ? M + __log2f(L) : -INFINITY;
    }
  }
}

// One warp per (request, head): merge the partitions of a decode row.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const Problem p) {
  const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.B * p.H) return;
  const int r = wid / p.H, h = wid % p.H;
  const int t0 = p.qsl[r];
  if (p.qsl[r + 1] - t0 != 1 || t0 < 0 || t0 >= p.T) return;
  const int S = p.splits;
  const int64_t prow = (static_cast<int64_t>(r) * p.H + h) * S;
  float M = -INFINITY;
  for (int sp = 0; sp < S; ++sp) M = fmaxf(M, p.lse_part[prow + sp]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int sp = 0; sp < S; ++sp) {
    const float l = p.lse_part[prow + sp];
    if (l == -INFINITY) continue;
    const float w = exp2f(l - Mu);
    L += w;
    const float* src = p.o_part + (prow + sp) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += w * src[e];
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (static_cast<int64_t>(t0) * p.H + h) * D + lane * PER;
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < PER; e += 2) {
    __nv_bfloat162 v = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
    *reinterpret_cast<__nv_bfloat162*>(out + e) = v;
  }
}

template <int D, bool FP8>
cudaError_t launch_decode_t(const Problem& p) {
  using C = DecodeCfg<D, FP8>;
  auto kern = decode_split_kernel<D, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  const float sl2 = p.scale * LOG2E * (FP8 ? p.k_scale : 1.f);
  const float out_scale = FP8 ? p.v_scale : 1.f;
  const long long items = static_cast<long long>(p.B) * p.Hkv * p.splits;
  if (items == 0) return cudaSuccess;
  kern<<<static_cast<unsigned>(items), DEC_WARPS * 32, C::SMEM_TOTAL, p.stream>>>(p, sl2, out_scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const Problem& p) {
  if (p.D == 128) return p.kv_dtype ? launch_decode_t<128, true>(p) : launch_decode_t<128, false>(p);
  return p.kv_dtype ? launch_decode_t<64, true>(p) : launch_decode_t<64, false>(p);
}

cudaError_t launch_combine(const Problem& p) {
  const long long rows = static_cast<long long>(p.B) * p.H;
  if (rows == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((rows + 3) / 4);
  if (p.D == 128)
    combine_kernel<128><<<grid, 128, 0, p.stream>>>(p);
  else
    combine_kernel<64><<<grid, 128, 0, p.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pattn
