// diffkv_decode.cu -- decode rows over a DiffKV cache on the tensor cores
// (sm_103a).
//
// "[vLLM] other attention backends", FlashAttention DiffKV: V has its own head
// size and the KV cache is asymmetric.  The layout read here (the reading the
// library takes; the page gives no shape) is one tensor
// [num_blocks][block_size][num_kv_heads][dk + dv], each row the token's K
// (dk elements) then its V (dv elements), 16-bit.  This kernel serves the rows
// with query_len == 1 (the prefill/decode split with threshold 1 of "[vLLM]
// Lightning & Linear Attention"); the generic kernel serves the others.
//
// One CTA per (decode request, KV head); head sizes that are multiples of 64
// (other sizes run on the generic kernel).  Two producer warps stage 16-key
// units through a ring of shared-memory stages, one TMA tensor copy per unit
// for the K part (warp 4) and one for the V part (warp 5) of 16 rows of the
// KV head: a copy holds its issuing warp for a while whatever its size, so a
// unit is two large copies rather than hundreds of 16-byte ones.  The tensor
// map views the cache as [rows][64-element chunks of a row][KV heads] and a
// box lands chunk-major, [chunk][row][128 bytes] with the 128-byte swizzle,
// so the ldmatrix reads of eight consecutive rows hit distinct bank groups.
// Rows at or past seq_len (stale slots of the last block, NaN included) are
// zeroed in shared memory before use.  Four consumer warps take the units in
// turn: S^T = K Q^T and O^T += V^T P^T on mma.sync m16n8k16 with the 16 keys
// (then the dv rows) as M and the query heads of the KV head as N, as the
// main decode kernel does; the online softmax keeps a lazy reference max, and
// the row sums come from one extra MMA against a ones tile.  At the end the
// four warps merge their (o, m, l) through shared memory and warp 0 writes the
// normalised rows.
#include "../../include/pattn.h"
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

constexpr int DKD_UNIT = 16;       // keys per unit
constexpr int DKD_CW = 4;          // consumer warps
constexpr int DKD_PW = 2;          // producer warps
constexpr int DKD_THREADS = (DKD_CW + DKD_PW) * 32;
constexpr float DKD_RESCALE_LOG2 = 8.0f;
constexpr unsigned DKD_FULL = 0xffffffffu;

__device__ __forceinline__ void ldsm_x2(unsigned addr, unsigned& r0, unsigned& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

// Byte offset of 16-byte unit u (of the row's 16-byte units) of row j in a
// chunk-major, 128-byte-swizzled box of 16 rows: chunk u / 8, unit u % 8
// swizzled with the row (line % 8 == row % 8 since a chunk holds 16 rows).
__device__ __forceinline__ int swz(int j, int u) {
  return (((u >> 3) << 4) + j) * 128 + (((u & 7) ^ (j & 7)) << 4);
}

// Ring depth for a stage of `stage` bytes: a multiple of the consumer warps
// (unit i goes to warp i % 4 and stage i % NST, so each stage is always read
// by one warp, which therefore never waits on a phase two ahead), 8 stages
// when they fit in ~96 KB (two CTAs per SM), else 4.
__host__ __device__ constexpr int dkd_stages(int stage) { return 8 * stage <= 98304 ? 8 : 4; }

// DV16 = dv / 16 output row tiles, NT = query-head tiles of 8 (G <= 8 * NT).
// kmap / vmap: boxes of 16 rows x all K (or V) chunks of one KV head.
template <int DV16, int NT, bool HALF>
__global__ void __launch_bounds__(DKD_THREADS, 2)
    diffkv_decode_kernel(const __grid_constant__ Problem p, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, int dk, float sl2) {
  constexpr int DV = DV16 * 16;
  extern __shared__ unsigned char smem_raw[];
  // the 128-byte swizzle is laid out from 1024-byte aligned boxes
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int KBYTES = DKD_UNIT * 2 * dk;       // K part of a stage
  const int STAGE = KBYTES + DKD_UNIT * 2 * DV;
  const int NST = dkd_stages(STAGE);
  const int QS = 2 * dk + 16;                 // q row stride in shared memory
  unsigned char* ring = smem;
  unsigned char* qs = smem + NST * STAGE;     // [NT * 8][QS]
  uint64_t* full = reinterpret_cast<uint64_t*>(qs + NT * 8 * QS);
  uint64_t* empty = full + NST;

  // CTA (g, rank * P + sp): partition sp of the KV head g of the request of
  // rank `rank`.  The KV heads of a request are neighbours in the grid, so
  // they read the rows of the same blocks (interleaved in memory) at about
  // the same time; requests run longest first (the order the clearing kernel
  // wrote), so the grid's ragged end holds the short ones.
  const int P = p.splits;
  const int rank = static_cast<int>(blockIdx.y) / P, sp = static_cast<int>(blockIdx.y) % P;
  // In a decode-only call the clearing kernel before this one may still be
  // running (this kernel is its programmatic dependent): wait for it before
  // the decode order, the status word and the counters it writes.
  if (p.pdl_wait) grid_dep_wait();
  const int r = p.decode_order ? p.decode_order[rank] : rank;
  const int g = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  unsigned* status = &p.hdr->status;
  const int t0 = p.qsl[r];
  if (p.qsl[r + 1] - t0 != 1) return;  // not a decode row: the generic kernel's
  const int s = p.seq_lens[r];
  const int64_t orow = (static_cast<int64_t>(t0) * p.H + static_cast<int64_t>(g) * G) * DV;
  if (s < 1 || s > p.mbps * p.bs || t0 < 0 || t0 >= p.T) {
    // bad metadata: reported, the rows (if inside out) written as zeros
    if (sp != 0) return;
    if (threadIdx.x == 0) flag_status(status, PATTN_DEV_BAD_METADATA);
    if (t0 >= 0 && t0 < p.T)
      for (int e = threadIdx.x; e < G * DV; e += DKD_THREADS) {
        if constexpr (HALF)
          static_cast<__half*>(p.out)[orow + e] = __float2half_rn(0.f);
        else
          static_cast<__nv_bfloat16*>(p.out)[orow + e] = __float2bfloat16_rn(0.f);
      }
    return;
  }
  // visible keys of the decode row (position s - 1): [k_lo, s); units of 16
  // keys from the 16-aligned key at or below k_lo (a unit never straddles a
  // block: block_size is a multiple of 16); partition sp takes a contiguous
  // run of ceil(n / P) of the row's n units
  const int k_lo = (p.window > 0) ? max(0, s - p.window) : 0;
  const int n_all = (s - (k_lo & ~(DKD_UNIT - 1)) + DKD_UNIT - 1) / DKD_UNIT;
  const int per = (n_all + P - 1) / P;
  const int u0 = (k_lo & ~(DKD_UNIT - 1)) + sp * per * DKD_UNIT;
  const int n_units = max(0, min(per, n_all - sp * per));

  if (threadIdx.x == 0) {
    for (int b = 0; b < NST; ++b) {
      mbar_init(&full[b], 2);  // the K and the V producer each post their bytes
      mbar_init(&empty[b], 1);
    }
    fence_mbar_init();
  }
  // q of the G heads (16-bit, rows G .. 8 NT - 1 zero)
  {
    const unsigned short* qg = static_cast<const unsigned short*>(p.q) +
                               (static_cast<int64_t>(t0) * p.H + static_cast<int64_t>(g) * G) * dk;
    const int per_row = dk / 8;  // 16-byte pieces of a q row
    for (int c = threadIdx.x; c < NT * 8 * per_row; c += DKD_THREADS) {
      const int h = c / per_row, j = c % per_row;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (h < G) v = *reinterpret_cast<const uint4*>(qg + static_cast<int64_t>(h) * dk + j * 8);
      *reinterpret_cast<uint4*>(qs + h * QS + j * 16) = v;
    }
  }
  __syncthreads();

  if (warp >= DKD_CW) {
    // ------------------------------------------------------------ producer warps
    // Warp 4 copies the K part and warp 5 the V part of each unit, one tensor
    // copy each, as soon as the unit's stage is free; each posts its bytes on
    // the stage's full barrier.  Block ids come 32 units at a time from one
    // coalesced load.
    const int kv = warp - DKD_CW;
    const CUtensorMap* map = kv ? &vmap : &kmap;
    const int chunk0 = kv ? dk / 64 : 0;
    const unsigned bytes = static_cast<unsigned>(kv ? STAGE - KBYTES : KBYTES);
    if (lane == 0) tma_prefetch_desc(map);
    const int* bt = p.block_table + static_cast<int64_t>(r) * p.bt_stride;
    int ok = 1, armed_end = 0;
    for (int base = 0; ok && base < n_units; base += 32) {
      int my_blk = 0;
      if (base + lane < n_units) {
        my_blk = bt[(u0 + (base + lane) * DKD_UNIT) / p.bs];
        if (my_blk < 0 || my_blk >= p.NB) {
          flag_status(status, PATTN_DEV_BAD_METADATA);
          my_blk = min(max(my_blk, 0), p.NB - 1);
        }
      }
      const int nb = min(32, n_units - base);
      for (int l = 0; l < nb; ++l) {
        const int blk = __shfl_sync(DKD_FULL, my_blk, l);
        if (lane == 0) {
          const int i = base + l, st = i % NST;
          if (i >= NST && !mbar_wait(&empty[st], ((i / NST) - 1) & 1, status, nullptr)) {
            ok = 0;
          } else {
            armed_end = i + 1;
            const int key0 = u0 + i * DKD_UNIT;
            mbar_arrive_expect_tx(&full[st], bytes);
            tma_load_4d(ring + st * STAGE + kv * KBYTES, map, &full[st], 0,
                        blk * p.bs + key0 % p.bs, chunk0, g);
          }
        }
        if (!__shfl_sync(DKD_FULL, ok, 0)) break;
      }
    }
    // After a wait gave up, no armed copy may still be writing shared memory
    // when the CTA exits (otherwise the consumers wait for every copy).  The
    // stage's phase also needs the other producer's bytes; if that warp gave
    // up first, this wait runs out (bounded) instead.
    if (!ok && lane == 0) drain_armed(full, NST, armed_end, -1, status);
    return;
  }

  // ---------------------------------------------------------------- consumer warps
  const int quad = lane >> 2, c4 = lane & 3;
  const int mi = lane >> 3;
  const int KU = dk / 8;  // 16-byte units of a K row
  const int s_row = (lane & 7) + ((mi & 1) << 3), s_csel = mi >> 1;  // K rows (A, non-trans)
  const int v_row = (lane & 7) + ((mi >> 1) << 3), v_csel = mi & 1;  // V rows (A, trans)
  const int src0 = 8 * c4 + (quad >> 1), src1 = src0 + 4;           // P^T gather
  const unsigned half_sel = (quad & 1) ? 0x7632u : 0x5410u;
  const unsigned qbase = smem_u32(qs) + (lane & 7) * QS + ((lane >> 3) & 1) * 16;

  float o[DV16][NT][4], o_l[NT][4], m_run[NT][2];
#pragma unroll
  for (int m = 0; m < DV16; ++m)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[m][nt][0] = o[m][nt][1] = o[m][nt][2] = o[m][nt][3] = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    o_l[nt][0] = o_l[nt][1] = o_l[nt][2] = o_l[nt][3] = 0.f;
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
  }

  for (int i = warp; i < n_units; i += DKD_CW) {
    const int st = i % NST;
    if (!__all_sync(DKD_FULL, mbar_wait(&full[st], (i / NST) & 1, status, nullptr))) break;
    unsigned char* stage = ring + st * STAGE;
    const unsigned sb = smem_u32(stage);
    const int key0 = u0 + i * DKD_UNIT;
    // Rows at or past seq_len may hold anything (NaN included): zero them
    // (only the last unit has any).
    if (key0 + DKD_UNIT > s) {
      const int units = KU + DV / 8;  // 16-byte units of a K + V row
      for (int c = lane; c < DKD_UNIT * units; c += 32) {
        const int j = c / units, u = c % units;
        if (key0 + j >= s) {
          unsigned char* dst = (u < KU) ? stage + swz(j, u) : stage + KBYTES + swz(j, u - KU);
          *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
      }
      // the stage is refilled by TMA (async proxy) after this warp releases it
      fence_proxy_async_smem();
      __syncwarp();
    }
    // S^T = K Q^T: M = the 16 keys, N = heads, K = dk (two accumulation chains)
    float sc[2][NT][4];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sc[ch][nt][0] = sc[ch][nt][1] = sc[ch][nt][2] = sc[ch][nt][3] = 0.f;
#pragma unroll 2
    for (int kk = 0; kk < dk / 16; ++kk) {
      unsigned a0, a1, a2, a3;
      ldsm_x4(sb + swz(s_row, 2 * kk + s_csel), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        unsigned b0, b1;
        ldsm_x2(qbase + nt * 8 * QS + kk * 32, b0, b1);
        mma_16816<HALF>(sc[kk & 1][nt], a0, a1, a2, a3, b0, b1);
      }
    }
    // mask (keys quad, quad + 8), log2 units, lazy reference max
    const int ka = key0 + quad, kb = ka + 8;
    const bool va = ka >= k_lo && ka < s, vb = kb >= k_lo && kb < s;
    float x[NT][4];
    bool grow = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v = sc[0][nt][e] + sc[1][nt][e];
        x[nt][e] = ((e < 2) ? va : vb) ? v * sl2 : -INFINITY;
        grow |= x[nt][e] > m_run[nt][e & 1] + DKD_RESCALE_LOG2;
      }
    if (__any_sync(DKD_FULL, grow)) {
      float alpha[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float mx = fmaxf(x[nt][h2], x[nt][2 + h2]);
          mx = fmaxf(mx, __shfl_xor_sync(DKD_FULL, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(DKD_FULL, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(DKD_FULL, mx, 16));
          const bool mv = mx > m_run[nt][h2] + DKD_RESCALE_LOG2;
          alpha[nt][h2] = !mv ? 1.f : (m_run[nt][h2] == -INFINITY) ? 0.f : fast_exp2(m_run[nt][h2] - mx);
          if (mv) m_run[nt][h2] = mx;
        }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) o_l[nt][e] *= alpha[nt][e & 1];
#pragma unroll
        for (int m = 0; m < DV16; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[m][nt][e] *= alpha[nt][e & 1];
      }
    }
    // P^T as the B operand of O^T += V^T P^T
    unsigned pb0[NT], pb1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float r0 = (m_run[nt][0] == -INFINITY) ? 0.f : m_run[nt][0];
      const float r1 = (m_run[nt][1] == -INFINITY) ? 0.f : m_run[nt][1];
      const unsigned lo = pack2<HALF>(fast_exp2(x[nt][0] - r0), fast_exp2(x[nt][1] - r1));
      const unsigned hi = pack2<HALF>(fast_exp2(x[nt][2] - r0), fast_exp2(x[nt][3] - r1));
      const unsigned x0 = __shfl_sync(DKD_FULL, lo, src0), x1 = __shfl_sync(DKD_FULL, lo, src1);
      const unsigned y0 = __shfl_sync(DKD_FULL, hi, src0), y1 = __shfl_sync(DKD_FULL, hi, src1);
      pb0[nt] = __byte_perm(x0, x1, half_sel);
      pb1[nt] = __byte_perm(y0, y1, half_sel);
    }
    const unsigned vb0 = sb + KBYTES;
#pragma unroll
    for (int m = 0; m < DV16; ++m) {
      unsigned a0, a1, a2, a3;
      ldsm_x4_t(vb0 + swz(v_row, 2 * m + v_csel), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816<HALF>(o[m][nt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
    }
    // row sums of the (rounded) weights: 1^T P^T
    constexpr unsigned ONES = HALF ? 0x3C003C00u : 0x3F803F80u;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_16816<HALF>(o_l[nt], ONES, ONES, ONES, ONES, pb0[nt], pb1[nt]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---------------------------------------------------------------- merge
  // Every unit has been read (its copies landed): the ring is free.  Warps
  // 1..3 hand (o, m, l) to warp 0 in the fragment layout.
  named_bar_sync(1, DKD_CW * 32);
  constexpr int MF = DV16 * NT * 4 + 4 * NT;  // floats per lane
  float* mb = reinterpret_cast<float*>(ring);
  if (warp > 0) {
    float* dst = mb + (warp - 1) * MF * 32 + lane;
    int idx = 0;
#pragma unroll
    for (int m = 0; m < DV16; ++m)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[32 * idx++] = o[m][nt][e];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        dst[32 * idx++] = m_run[nt][h2];
        dst[32 * idx++] = o_l[nt][h2];
      }
  }
  named_bar_sync(1, DKD_CW * 32);
  if (warp != 0) return;
  float l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    l_run[nt][0] = o_l[nt][0];
    l_run[nt][1] = o_l[nt][1];
  }
  for (int w = 1; w < DKD_CW; ++w) {
    const float* src = mb + (w - 1) * MF * 32 + lane;
    float a_self[NT][2], a_other[NT][2];
    int idx = DV16 * NT * 4;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const float m2 = src[32 * idx++], l2 = src[32 * idx++];
        const float mn = fmaxf(m_run[nt][h2], m2);
        const float mu = (mn == -INFINITY) ? 0.f : mn;
        a_self[nt][h2] = fast_exp2(m_run[nt][h2] - mu);
        a_other[nt][h2] = fast_exp2(m2 - mu);
        l_run[nt][h2] = l_run[nt][h2] * a_self[nt][h2] + l2 * a_other[nt][h2];
        m_run[nt][h2] = mn;
      }
    idx = 0;
#pragma unroll
    for (int m = 0; m < DV16; ++m)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[m][nt][e] = o[m][nt][e] * a_self[nt][e & 1] + src[32 * idx++] * a_other[nt][e & 1];
  }
  if (P == 1) {
    // normalise (the head's sink joins the normaliser) and write the G rows
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int head = nt * 8 + 2 * c4 + (e & 1);
        if (head >= G) continue;
        const float L = l_run[nt][e & 1] + sink_term(p.sinks, g * G + head, m_run[nt][e & 1]);
        const float inv = (L > 0.f) ? 1.f / L : 0.f;
        const int64_t ob = orow + static_cast<int64_t>(head) * DV + quad + ((e & 2) ? 8 : 0);
#pragma unroll
        for (int m = 0; m < DV16; ++m) {
          const float val = o[m][nt][e] * inv;
          if constexpr (HALF)
            static_cast<__half*>(p.out)[ob + 16 * m] = __float2half_rn(val);
          else
            static_cast<__nv_bfloat16*>(p.out)[ob + 16 * m] = __float2bfloat16_rn(val);
        }
      }
    return;
  }
  // ---------------------------------------------------------------- partitions
  // The partition's normalised o (fp32) and its lse = m + log2 l go to the
  // workspace, [r][h][P][DV] and [r][h][P]; the CTA that completes the count
  // of its (request, KV head) merges the P partitions by log-sum-exp ("RBLN
  // Attention modes", flash attention: partition results merged with online
  // softmax), an empty one (lse = -inf) weighing 0.
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int head = nt * 8 + 2 * c4 + (e & 1);
      if (head >= G) continue;
      const float L = l_run[nt][e & 1], M = m_run[nt][e & 1];
      const float inv = (L > 0.f) ? 1.f / L : 0.f;
      const int64_t prow = (static_cast<int64_t>(r) * p.H + g * G + head) * P + sp;
#pragma unroll
      for (int m = 0; m < DV16; ++m)
        p.o_part[prow * DV + 16 * m + quad + ((e & 2) ? 8 : 0)] = o[m][nt][e] * inv;
      if (quad == 0 && (e & 2) == 0) p.lse_part[prow] = (L > 0.f) ? M + __log2f(L) : -INFINITY;
    }
  // publish (release, cumulative over the warp's stores ordered by the fence
  // and the warp barrier) and count; the add that completes the count
  // acquires the other partitions'
  __threadfence();
  __syncwarp();
  unsigned last = 0;
  if (lane == 0) {
    unsigned* cnt = p.counters + static_cast<int64_t>(r) * p.Hkv + g;
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(cnt) : "memory");
    last = (prev == static_cast<unsigned>(P - 1)) ? 1u : 0u;
    if (last) *cnt = 0u;  // every partition has counted
  }
  if (!__shfl_sync(DKD_FULL, last, 0)) return;
  for (int head = 0; head < G; ++head) {
    const int64_t prow0 = (static_cast<int64_t>(r) * p.H + g * G + head) * P;
    float w0 = (lane < P) ? __ldcg(p.lse_part + prow0 + lane) : -INFINITY;
    float w1 = (lane + 32 < P) ? __ldcg(p.lse_part + prow0 + lane + 32) : -INFINITY;
    float M = fmaxf(w0, w1);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(DKD_FULL, M, o2));
    const float Mu = (M == -INFINITY) ? 0.f : M;
    w0 = (w0 == -INFINITY) ? 0.f : exp2f(w0 - Mu);
    w1 = (w1 == -INFINITY) ? 0.f : exp2f(w1 - Mu);
    float L = w0 + w1;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(DKD_FULL, L, o2);
    L += sink_term(p.sinks, g * G + head, Mu);
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    float acc[DV / 32];
#pragma unroll
    for (int c = 0; c < DV / 32; ++c) acc[c] = 0.f;
    for (int q = 0; q < P; ++q) {
      const float w = __shfl_sync(DKD_FULL, q < 32 ? w0 : w1, q & 31);
      const float* src = p.o_part + (prow0 + q) * DV + lane;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) acc[c] += w * __ldcg(src + 32 * c);
    }
    const int64_t ob = orow + static_cast<int64_t>(head) * DV + lane;
#pragma unroll
    for (int c = 0; c < DV / 32; ++c) {
      if constexpr (HALF)
        static_cast<__half*>(p.out)[ob + 32 * c] = __float2half_rn(acc[c] * inv);
      else
        static_cast<__nv_bfloat16*>(p.out)[ob + 32 * c] = __float2bfloat16_rn(acc[c] * inv);
    }
  }
}

template <int DV16, int NT, bool HALF>
cudaError_t launch_t(const Problem& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int dk) {
  constexpr int DV = DV16 * 16;
  const int stage = DKD_UNIT * 2 * (dk + DV);
  const int nst = dkd_stages(stage);
  const size_t ring = static_cast<size_t>(nst) * stage;
  const size_t merge = static_cast<size_t>(DKD_CW - 1) * (DV16 * NT * 4 + 4 * NT) * 32 * 4;
  const size_t smem = (ring > merge ? ring : merge) + static_cast<size_t>(NT) * 8 * (2 * dk + 16) +
                      2 * nst * 8 + 1024;
  auto k = diffkv_decode_kernel<DV16, NT, HALF>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const float sl2 = fmaxf(p.scale * LOG2E, 1e-30f);
  const dim3 grid(static_cast<unsigned>(p.Hkv),
                  static_cast<unsigned>(p.B) * static_cast<unsigned>(p.splits));
  if (p.pdl_launch) {
    // programmatic dependent of the previous kernel in the stream
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(DKD_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = p.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, p, kmap, vmap, dk, sl2);
  }
  k<<<grid, DKD_THREADS, smem, p.stream>>>(p, kmap, vmap, dk, sl2);
  return cudaGetLastError();
}

template <int NT, bool HALF>
cudaError_t launch_nt(const Problem& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int dk,
                      int dv) {
  switch (dv / 16) {
    case 4: return launch_t<4, NT, HALF>(p, kmap, vmap, dk);
    case 8: return launch_t<8, NT, HALF>(p, kmap, vmap, dk);
    case 12: return launch_t<12, NT, HALF>(p, kmap, vmap, dk);
    case 16: return launch_t<16, NT, HALF>(p, kmap, vmap, dk);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool diffkv_decode_supported(int dk, int dv) { return dk % 64 == 0 && dv % 64 == 0; }

// The decode rows of a DiffKV batch (dk, dv multiples of 64 up to 256; G <= 16).
cudaError_t launch_diffkv_decode(const Problem& p, int dk, int dv) {
  if (p.B == 0 || p.T == 0) return cudaSuccess;
  CUtensorMap kmap, vmap;
  if (!encode_diffkv_map(&kmap, p.kv, p.kv_dtype, dk, dv, p.Hkv, p.bs, p.NB, dk / 64) ||
      !encode_diffkv_map(&vmap, p.kv, p.kv_dtype, dk, dv, p.Hkv, p.bs, p.NB, dv / 64))
    return cudaErrorInvalidValue;
  const bool half = p.kv_dtype == PATTN_KV_F16;
  if (p.G <= 8)
    return half ? launch_nt<1, true>(p, kmap, vmap, dk, dv) : launch_nt<1, false>(p, kmap, vmap, dk, dv);
  return half ? launch_nt<2, true>(p, kmap, vmap, dk, dv) : launch_nt<2, false>(p, kmap, vmap, dk, dv);
}

}  // namespace pattn
