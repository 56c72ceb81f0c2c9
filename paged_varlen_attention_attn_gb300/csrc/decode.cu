// decode.cu -- split-KV decode kernel and log-sum-exp combine (sm_103a).
//
// Decode rows (query_len == 1; the prefill/decode split with threshold 1 of
// "[vLLM] Lightning & Linear Attention") are bound by reading K/V from HBM:
// each KV byte feeds 2G (bf16) FLOPs, far below the tensor ridge.  One CTA
// takes one (request, group of HG KV heads, partition) item, so the G query
// heads of a KV head share every page it reads (FlashAttentionImpl's
// num_queries_per_kv).  The partition is a run of whole KV blocks ("RBLN
// Attention modes": flash attention processes the cache by partitions and
// merges them with online softmax); partial results go to the workspace as
// (o_p, lse_p) and the last CTA of each (request, group) to finish merges
// them, or the CTA writes the output directly when there is one partition.
//
// Data path: a producer warp streams 16-key units through a ring of
// shared-memory stages; one unit is 16 rows of all HG heads of the group, K
// and V, fetched with two TMA tensor copies (a 5-D map for 16-bit data, whose
// box spans both 64-element halves of the head dimension, a 4-D map for e4m3;
// 128-byte swizzle so ldmatrix reads are conflict-free).  One unit never
// straddles a KV block because block_size % 16 == 0.  Few, large copies keep
// many bytes in flight per SM with little issue work, which is what a
// bandwidth-bound stream needs.  Consumer warps compute S^T = K Q^T and
// O^T += V^T P^T on mma.sync m16n8k16 with the keys (and d) as the M rows and
// the G heads as N, so no MMA rows are wasted at small G; the tensor work is
// far below what HBM allows either way.  At G <= 8 two warps serve each KV
// head, taking the partition's units in turn, and merge their (o, m, l) at the
// end, which doubles the warps that hide load latency.  e4m3 K and V
// fragments are widened to f16 in registers, two codes per conversion
// instruction (exact: every e4m3 value is an f16 value); the per-tensor
// scales are folded into the softmax scale (K) and the final normalisation
// (V).
#include "../../include/pattn.h"
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

// A CTA serves one (request, group of HG KV heads, partition) item: WPH
// consumer warps per KV head, which take the partition's 16-key units in turn
// and merge their partial results at the end, plus one producer warp.
constexpr int UNIT = 16;  // keys per unit
constexpr int U = 1;      // units a consumer warp takes per softmax step
// lazy rescale threshold of the online softmax (log2 units): weights stay below 2^8
constexpr float RESCALE_LOG2 = 8.0f;

// KV heads per CTA: the largest of 4 / 2 / 1 that divides num_kv_heads and
// keeps one stage (K + V of 16 keys of the group) within 16 KB, so the ring
// holds six or more stages in ~96 KB.
__host__ __device__ constexpr int decode_head_group(int Hkv, int D, bool fp8) {
  return (Hkv % 4 == 0 && 4 * 2 * 16 * D * (fp8 ? 1 : 2) <= 16384) ? 4
         : (Hkv % 2 == 0) ? 2
                          : 1;
}

template <int D, bool FP8, int NT, int HG, int WPH>
struct DecodeCfg {
  static constexpr int ES = FP8 ? 1 : 2;
  static constexpr int RAW_ROW = D * ES;            // bytes of one key row of one head
  static constexpr int RAW_UNIT = UNIT * RAW_ROW;   // bytes of one head's K (or V) unit
  static constexpr int KV_UNIT = HG * RAW_UNIT;     // K (or V) of the whole head group
  static constexpr int STAGE = 2 * KV_UNIT;         // K + V of the head group
  // Ring depth: as many stages as fit in ~96 KB (two CTAs per SM), at most 8,
  // rounded down to a multiple of SLOTS = U x WPH.  Unit i goes to warp slot
  // (i / U) % WPH and stage i % NST; with NST a multiple of SLOTS every use of
  // a stage belongs to one slot, so a warp waiting on a stage's full barrier
  // has itself consumed the stage's previous phase and is never two phases
  // ahead of it (where a parity wait would pass at once).
  static constexpr int SLOTS = U * WPH;
  static constexpr int NST_FIT = (96 * 1024) / STAGE;
  static constexpr int NST_CAP = NST_FIT > 8 ? 8 : NST_FIT;
  static constexpr int NST = (NST_CAP / SLOTS) * SLOTS < 2 * SLOTS ? 2 * SLOTS : (NST_CAP / SLOTS) * SLOTS;
  static_assert(NST % SLOTS == 0, "each stage must belong to one warp slot");
  static constexpr int NW = HG * WPH;               // consumer warps
  // Partial state one warp hands over for the merge: o, m, l per lane.
  static constexpr int MERGE_FLOATS = (D / 16) * NT * 4 + 4 * NT;
  static constexpr int MERGE_BYTES = (WPH - 1) * HG * MERGE_FLOATS * 32 * 4;
  static constexpr int RING_BYTES = NST * STAGE;
  static constexpr int BAR_OFF = RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES;
  // block ids of the next 32 units, one buffer per producer warp
  static constexpr int ID_OFF = BAR_OFF + 2 * NST * 8 <= BAR_OFF + 256 ? BAR_OFF + 256 : -1;
  static_assert(ID_OFF > 0, "barriers fit in 256 bytes");
  static constexpr int SMEM = ID_OFF + 2 * 32 * 4 + 1024;
  // consumer warps, then two producer warps (K copies, V copies)
  static constexpr int THREADS = (NW + 2) * 32;
};

// e4m3 -> f16 widening with the hardware pair conversion: exact (every e4m3
// value, subnormals included, is an f16 value) and NaN codes stay NaN.
// The four codes of x as two f16x2: (bytes 0, 1) -> lo, (bytes 2, 3) -> hi.
// The 16-bit halves feed the pair conversions directly.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(unsigned x, unsigned& lo, unsigned& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

// Byte offset of 16-byte chunk c of row j of head hh in a K (or V) unit as
// TMA lays it down.  16-bit data: [d half][head][row][128 bytes], 128-byte
// swizzle (chunk index XOR line % 8, and line % 8 == row % 8 because each
// head block holds 16 rows).  e4m3 rows of 128 bytes: [head][row][128 B],
// same swizzle; 64-byte e4m3 rows: [head][row][64 B], no swizzle.
template <int D, bool FP8, int HG>
__device__ __forceinline__ int raw_off(int hh, int j, int c) {
  if constexpr (FP8 && D == 64) {
    return (hh * UNIT + j) * 64 + (c << 4);
  } else if constexpr (FP8) {
    return (hh * UNIT + j) * 128 + ((c ^ (j & 7)) << 4);
  } else {
    return (((c >> 3) * HG + hh) * UNIT + j) * 128 + (((c & 7) ^ (j & 7)) << 4);
  }
}

// The D / 8 bytes of e4m3 V row j of head hh that lane group q owns
// (bytes q * D/8 .. + D/8 of the row), as D / 32 words.
template <int D, int HG>
__device__ __forceinline__ void load_v_bytes(const unsigned char* sv, int hh, int j, int q,
                                             unsigned (&w)[D / 32]) {
  if constexpr (D == 128) {
    const uint4 x = *reinterpret_cast<const uint4*>(sv + raw_off<D, true, HG>(hh, j, q));
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
  } else {
    const uint2 x = *reinterpret_cast<const uint2*>(sv + (hh * UNIT + j) * 64 + q * 8);
    w[0] = x.x; w[1] = x.y;
  }
}

// One warp merges the S partitions (S <= 64) of NH decode rows (request r,
// heads h .. h + NH - 1): out = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M),
// M = max_p lse_p (log2 units); an empty partition (lse_p = -inf) weighs 0.
// Lanes hold the partitions' lse (two each), the max and the weight sum are
// warp reductions, and the loads of all partitions and all NH rows are
// independent, so the merge costs a few memory round trips, not S * NH of
// them.  The partials were written by other CTAs: they are read past L1.
template <int D, int NH, bool HALF>
__device__ __forceinline__ void merge_partitions(const Problem& p, int r, int h, int t0, int lane) {
  const int S = p.splits;
  constexpr int PER = D / 32;
  float w0[NH], w1[NH], inv[NH], acc[NH][PER], Mx[NH];
#pragma unroll
  for (int k = 0; k < NH; ++k) {
    const int64_t prow = (static_cast<int64_t>(r) * p.H + h + k) * S;
    w0[k] = (lane < S) ? __ldcg(p.lse_part + prow + lane) : -INFINITY;
    w1[k] = (lane + 32 < S) ? __ldcg(p.lse_part + prow + lane + 32) : -INFINITY;
  }
#pragma unroll
  for (int k = 0; k < NH; ++k) {
    float M = fmaxf(w0[k], w1[k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Mu = (M == -INFINITY) ? 0.f : M;
    Mx[k] = Mu;
    w0[k] = (w0[k] == -INFINITY) ? 0.f : exp2f(w0[k] - Mu);
    w1[k] = (w1[k] == -INFINITY) ? 0.f : exp2f(w1[k] - Mu);
    float L = w0[k] + w1[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    // a final output (not a partial for a later merge) includes the sink
    if (!p.o32) L += sink_term(p.sinks, h + k, Mu);
    inv[k] = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[k][e] = 0.f;
  }
#pragma unroll 2
  for (int sp = 0; sp < S; ++sp) {
#pragma unroll
    for (int k = 0; k < NH; ++k) {
      const float w = __shfl_sync(0xffffffffu, sp < 32 ? w0[k] : w1[k], sp & 31);
      const float* src = p.o_part + ((static_cast<int64_t>(r) * p.H + h + k) * S + sp) * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
        acc[k][0] += w * v.x; acc[k][1] += w * v.y; acc[k][2] += w * v.z; acc[k][3] += w * v.w;
      } else {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
        acc[k][0] += w * v.x; acc[k][1] += w * v.y;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < NH; ++k) {
    const int64_t o0 = (static_cast<int64_t>(t0) * p.H + h + k) * D + lane * PER;
    if (p.o32) {
#pragma unroll
      for (int e = 0; e < PER; ++e) p.o32[o0 + e] = acc[k][e] * inv[k];
      if (lane == 0) p.lse32[o0 / D] = (inv[k] > 0.f) ? Mx[k] - __log2f(inv[k]) : -INFINITY;
    } else {
#pragma unroll
      for (int e = 0; e < PER; e += 2)
        *(static_cast<unsigned*>(p.out) + (o0 + e) / 2) =
            pack2<HALF>(acc[k][e] * inv[k], acc[k][e + 1] * inv[k]);
    }
  }
}

// HALF: q, a 16-bit cache and out are f16 (else bf16; an e4m3 cache goes with
// bf16 q and out).
template <int D, bool FP8, int NT, int HG, int WPH, bool HALF>
__global__ void __launch_bounds__(DecodeCfg<D, FP8, NT, HG, WPH>::THREADS, WPH > 1 ? 2 : 1)
    decode_split_kernel(const Problem p, const __grid_constant__ CUtensorMap kvmap, float sl2,
                        float out_scale) {
  using C = DecodeCfg<D, FP8, NT, HG, WPH>;
  constexpr int NST = C::NST;
  extern __shared__ unsigned char smem_raw[];
  // TMA's 128-byte swizzle is laid out from 1024-byte aligned boxes
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.splits;
  const int n_groups = p.Hkv / HG;
  const int item = blockIdx.x;
  const int sp = item % S;
  const int grp = (item / S) % n_groups;
  // Requests are taken longest first (the order the kernel before this one
  // wrote), so the grid's ragged end holds the short partitions.  In a
  // decode-only call that kernel may still be running: wait for it (it also
  // clears the status word and the counters).
  if (p.pdl_wait) grid_dep_wait();
  const int rank = item / (S * n_groups);
  const int r = p.decode_order ? p.decode_order[rank] : rank;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  const int hh = warp % HG, wslot = warp / HG;  // consumer: head in the group, unit slot
  const int g = grp * HG + hh;                  // this consumer warp's KV head
  const int quad = lane >> 2, c4 = lane & 3;    // fragment row / column group

  const int t0 = p.qsl[r];
  const int q_len = p.qsl[r + 1] - t0;
  if (q_len != 1) {
    // A call declared decode-only (max_query_len <= 1) runs no other kernel
    // over its requests: a longer one is bad metadata, reported and zeroed
    // here (once, clamped to the output).  A decode-rows-only call leaves
    // such requests to another call.
    if (p.max_q <= 1 && !p.decode_rows_only && q_len != 0 && grp == 0 && sp == 0) {
      if (threadIdx.x == 0) flag_status(&p.hdr->status, PATTN_DEV_BAD_METADATA);
      const int64_t a = static_cast<int64_t>(max(0, t0)) * p.H * D;
      const int64_t b = static_cast<int64_t>(min(p.T, t0 + max(q_len, 0))) * p.H * D;
      if (p.o32) {
        for (int64_t e = a + threadIdx.x; e < b; e += blockDim.x) p.o32[e] = 0.f;
        for (int64_t e = a / D + threadIdx.x; e < b / D; e += blockDim.x) p.lse32[e] = -INFINITY;
      } else {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
        for (int64_t e = a + threadIdx.x; e < b; e += blockDim.x) out[e] = __float2bfloat16_rn(0.f);
      }
    }
    return;
  }
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

  // Units (16 keys of all HG heads) of this item.
  const int u_begin = kb / UNIT;
  const int u_end = (ke + UNIT - 1) / UNIT;
  const int n_units = (ke > kb) ? (u_end - u_begin) : 0;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);   // [NST]
  uint64_t* empty = full + NST;                                       // [NST]
  if (threadIdx.x == 0) {
    for (int b = 0; b < NST; ++b) {
      mbar_init(&full[b], 2);  // the K and the V producer each post their bytes
      mbar_init(&empty[b], HG);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp >= C::NW) {
    // ------------------------------------------------------------ producer warps
    // Warp NW copies the K rows of each unit (16 keys of all HG heads), warp
    // NW + 1 the V rows, each as one tensor copy per unit, as soon as the
    // consumers release the stage; each posts its own bytes on the stage's
    // full barrier.  A warp issues copies one after another (a copy holds
    // its issuing warp for a while), so two warps double the copy rate.
    // Block ids are read 32 units at a time (one coalesced load) into a
    // per-warp buffer; lane 0 then issues those units' copies.
    const int kv = warp - C::NW;
    int* ids = reinterpret_cast<int*>(smem + C::ID_OFF) + kv * 32;
    if (lane == 0) tma_prefetch_desc(&kvmap);
    const int* bt = p.block_table + static_cast<int64_t>(r) * p.bt_stride;
    int ok = 1;
    int armed_end = 0;  // units [0, armed_end) had this warp's bytes posted
#ifdef PATTN_WAIT_TEST
    // wait-test build: this unit posts no bytes and issues no copy, so the
    // consumers' wait for it runs out
    const int skip_pos = (p.test_skip == 2 && blockIdx.x == 0) ? 0 : -1;
#else
    constexpr int skip_pos = -1;
#endif
    for (int base = 0; ok && base < n_units; base += 32) {
      const int gu = base + lane;
      int blk = 0;
      if (gu < n_units) {
        const int key0 = (u_begin + gu) * UNIT;
        blk = bt[p.bs_shift >= 0 ? (key0 >> p.bs_shift) : (key0 / p.bs)];
        if (blk < 0 || blk >= p.NB) {
          flag_status(status, PATTN_DEV_BAD_METADATA);
          blk = min(max(blk, 0), p.NB - 1);
        }
      }
      ids[lane] = blk;
      __syncwarp();
      if (lane == 0) {
        const int nb = min(32, n_units - base);
        for (int l = 0; l < nb; ++l) {
          const int i = base + l, st = i % NST;
          if (i >= NST && !mbar_wait(&empty[st], ((i / NST) - 1) & 1, status, nullptr)) {
            ok = 0;
            break;
          }
          if (i == skip_pos) continue;
          armed_end = i + 1;
          const int key0 = (u_begin + i) * UNIT;
          const int slot = p.bs_shift >= 0 ? (key0 & (p.bs - 1)) : (key0 % p.bs);
          unsigned char* dst = smem + st * C::STAGE + kv * C::KV_UNIT;
          mbar_arrive_expect_tx(&full[st], C::KV_UNIT);
          if constexpr (FP8)
            tma_load_4d(dst, &kvmap, &full[st], 0, slot, grp * HG, kv * p.NB + ids[l]);
          else
            tma_load_5d(dst, &kvmap, &full[st], 0, slot, grp * HG, 0, kv * p.NB + ids[l]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();
    }
    // A wait gave up: no copy armed here may still be writing shared memory
    // when the CTA exits.  (Otherwise the consumers wait for every copy.)  The
    // stage's phase also needs the other producer's bytes; if that warp gave
    // up first, this wait runs out (bounded) instead.
    if (!ok && lane == 0) drain_armed(full, NST, armed_end, skip_pos, status);
    return;  // nothing after this needs the producers
  }

  // ---------------------------------------------------------------- consumer warps
  // Q^T in registers.  S^T = K Q^T: the B operand (16 d x 8 heads, "col") of
  // k-step kk and head tile nt is Q[head][d] at head = nt*8 + quad.  For
  // 16-bit K, d = 16kk + 2*c4 (+1, +8, +9).  For e4m3 K the d axis is permuted
  // (the same permutation on Q and K leaves every dot product unchanged) so
  // each lane reads its K bytes contiguously and widens whole words: k-step
  // kk, fragment columns 2*c4, 2*c4+1, 2*c4+8, 2*c4+9 map to d = base,
  // base + 1, base + 2, base + 3 with base = c4*D/4 + 4kk (the two 16-bit
  // halves of the word holding d = base..base+3).  There the f16 MMAs take q
  // in f16: each head's row is first scaled by the power of two sc that puts
  // its largest magnitude in [2^7, 2^8), so no bf16 value leaves f16's range
  // (exact down to 2^-21 of the row maximum), and its scores are scaled back
  // by 1 / sc with the score scale.
  unsigned qb[D / 16][NT][2];
  float sl2h[NT][2];  // score scale of the lane's head columns 2*c4, 2*c4 + 1
  {
    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                (static_cast<int64_t>(t0) * p.H + g * G) * D;
    if constexpr (FP8) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int head = nt * 8 + quad;
        // this lane's D/4 values of the head's row: d = c4*D/4 + 8i .. + 7 in w[i]
        uint4 w[D / 32];
#pragma unroll
        for (int i = 0; i < D / 32; ++i)
          w[i] = (head < G) ? *reinterpret_cast<const uint4*>(qrow + head * D + c4 * (D / 4) + 8 * i)
                            : make_uint4(0, 0, 0, 0);
        // the row's largest magnitude over its four lanes (bf16 magnitudes
        // compare as unsigned integers once the sign bit is cleared)
        unsigned m = 0;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const unsigned v[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) m = max(m, max(v[e] & 0x7fffu, (v[e] >> 16) & 0x7fffu));
        }
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        float sc, inv;
        split_scale(static_cast<int>(m >> 7), sc, inv);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            // d = base + 2e and base + 2e + 1 (word 2kk + e of the lane's range)
            const uint4& wi = w[(2 * kk + e) >> 2];
            const int c = (2 * kk + e) & 3;
            const unsigned x = c == 0 ? wi.x : c == 1 ? wi.y : c == 2 ? wi.z : wi.w;
            qb[kk][nt][e] = pack2<true>(__uint_as_float(x << 16) * sc,
                                        __uint_as_float(x & 0xffff0000u) * sc);
          }
        // the scales of the lane's output head columns (kept normal, so that
        // a masked score still maps to -inf)
        const float i0 = __shfl_sync(0xffffffffu, inv, (2 * c4) * 4);
        const float i1 = __shfl_sync(0xffffffffu, inv, (2 * c4 + 1) * 4);
        sl2h[nt][0] = fmaxf(sl2 * i0, 1e-37f);
        sl2h[nt][1] = fmaxf(sl2 * i1, 1e-37f);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int head = nt * 8 + quad;
            const int d = kk * 16 + 2 * c4 + e * 8;
            qb[kk][nt][e] = (head < G) ? *reinterpret_cast<const unsigned*>(qrow + head * D + d) : 0u;
          }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sl2h[nt][0] = sl2h[nt][1] = sl2;
    }
  }
  float o[D / 16][NT][4];
#pragma unroll
  for (int m = 0; m < D / 16; ++m)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[m][nt][0] = o[m][nt][1] = o[m][nt][2] = o[m][nt][3] = 0.f;
  // reference max of heads nt*8 + 2*c4 + h2 (identical across the lanes of
  // a column group), and the row sums of the weights, accumulated by MMAs in
  // the output fragment layout (every row of o_l holds the sums)
  float m_run[NT][2], l_run[NT][2], o_l[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    o_l[nt][0] = o_l[nt][1] = o_l[nt][2] = o_l[nt][3] = 0.f;
  }

  const int kmin = kb, kmax = ke;
  // ldmatrix lane addressing (matrix index = lane >> 3)
  const int mi = lane >> 3;
  const int s_row = (lane & 7) + ((mi & 1) << 3), s_csel = mi >> 1;    // K, non-transposed
  const int v_row = (lane & 7) + ((mi >> 1) << 3), v_csel = mi & 1;    // V, transposed
  // P^T gather: source lanes and half selector for this lane's B fragment
  const int src0 = 8 * c4 + (quad >> 1), src1 = src0 + 4;
  const unsigned half_sel = (quad & 1) ? 0x7632u : 0x5410u;

  // Each step takes U consecutive units (U x 16 keys): the scores of all of
  // them, one online-softmax update over their keys (the max and sum
  // reductions are shared), then P V for each.  Unit i sits in stage i % NST
  // and belongs to warp slot (i / U) % WPH.
  for (int i0 = wslot * U; i0 < n_units; i0 += WPH * U) {
    const int nu = min(U, n_units - i0);
    bool landed = true;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (u < nu) landed &= mbar_wait(&full[(i0 + u) % NST], ((i0 + u) / NST) & 1, status, nullptr);
    if (!__all_sync(0xffffffffu, landed)) break;
    const int key_base = (u_begin + i0) * UNIT;
    // Rows at or past seq_len may hold anything (NaN included): zero this
    // head's rows (only the partition's last unit can have any).
    if (key_base + nu * UNIT > s) {
      const int u = nu - 1;
      unsigned char* sk = smem + ((i0 + u) % NST) * C::STAGE;
      unsigned char* sv = sk + C::KV_UNIT;
      const int key0 = key_base + u * UNIT;
      constexpr int CH_ROW = C::RAW_ROW / 16;
      for (int c = lane; c < UNIT * CH_ROW; c += 32) {
        const int j = c / CH_ROW, cc = c % CH_ROW;
        if (key0 + j >= s) {
          *reinterpret_cast<uint4*>(sk + raw_off<D, FP8, HG>(hh, j, cc)) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(sv + raw_off<D, FP8, HG>(hh, j, cc)) = make_uint4(0, 0, 0, 0);
        }
      }
      // the stage is refilled by TMA (async proxy) after this warp releases it
      fence_proxy_async_smem();
      __syncwarp();
    }

    // S^T = K Q^T for the 16 keys of each unit: M = keys, N = heads, in two
    // independent accumulation chains per unit (even / odd k-steps).
    float sc[U][2][NT][4];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          sc[u][ch][nt][0] = sc[u][ch][nt][1] = sc[u][ch][nt][2] = sc[u][ch][nt][3] = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (u >= nu) break;
      const unsigned char* sk = smem + ((i0 + u) % NST) * C::STAGE;
      if constexpr (FP8) {
        // K fragments straight from the e4m3 bytes: this lane's D/4 bytes of
        // key rows quad and quad + 8, widened in registers.
        constexpr int CPL = D / 64;  // 16-byte chunks per lane per row
        uint4 kr[2][CPL];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
#pragma unroll
          for (int q = 0; q < CPL; ++q)
            kr[hr][q] = *reinterpret_cast<const uint4*>(sk + raw_off<D, FP8, HG>(hh, quad + 8 * hr, c4 * CPL + q));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint4& ra = kr[0][kk >> 2];
          const uint4& rb = kr[1][kk >> 2];
          const unsigned w0 = (kk & 3) == 0 ? ra.x : (kk & 3) == 1 ? ra.y : (kk & 3) == 2 ? ra.z : ra.w;
          const unsigned w1 = (kk & 3) == 0 ? rb.x : (kk & 3) == 1 ? rb.y : (kk & 3) == 2 ? rb.z : rb.w;
          unsigned a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(w0, a0, a2);  // key quad:     d base, base + 1 | base + 2, base + 3
          e4m3x4_to_f16x2x2(w1, a1, a3);  // key quad + 8
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816<true>(sc[u][kk & 1][nt], a0, a1, a2, a3, qb[kk][nt][0], qb[kk][nt][1]);
        }
      } else {
        const unsigned sk_a = smem_u32(sk);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          unsigned a0, a1, a2, a3;
          ldsm_x4(sk_a + raw_off<D, FP8, HG>(hh, s_row, 2 * kk + s_csel), a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816<HALF>(sc[u][kk & 1][nt], a0, a1, a2, a3, qb[kk][nt][0], qb[kk][nt][1]);
        }
      }
    }

    // Mask (keys quad and quad + 8 of each unit) and scale to log2 units.
    // Online softmax with a lazy reference max per head: the reference moves
    // only when a score exceeds it by more than 2^RESCALE_LOG2, so the common
    // step needs no cross-lane reduction and the weights 2^(x - ref) stay
    // below 2^RESCALE_LOG2.  O and the row sums (accumulated by the same MMAs)
    // are relative to the same reference, so the final O / l is exact.
    float x[U][NT][4];
    bool grow = false;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int ka = key_base + u * UNIT + quad, kb2 = ka + 8;
      const bool va = ka >= kmin && ka < kmax, vb = kb2 >= kmin && kb2 < kmax;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v = sc[u][0][nt][e] + sc[u][1][nt][e];
          x[u][nt][e] = ((e < 2) ? va : vb) ? v * sl2h[nt][e & 1] : -INFINITY;
          grow |= x[u][nt][e] > m_run[nt][e & 1] + RESCALE_LOG2;
        }
    }
    if (__any_sync(0xffffffffu, grow)) {
      // A head column's reference moves to its exact running max (the same in
      // the 8 lanes of the column after the reduction) when that max exceeds
      // it by more than the threshold; O and the sums are rescaled.
      float alpha[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float mx = fmaxf(x[0][nt][h2], x[0][nt][2 + h2]);
#pragma unroll
          for (int u = 1; u < U; ++u) mx = fmaxf(mx, fmaxf(x[u][nt][h2], x[u][nt][2 + h2]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const bool mv = mx > m_run[nt][h2] + RESCALE_LOG2;
          alpha[nt][h2] = !mv ? 1.f : (m_run[nt][h2] == -INFINITY) ? 0.f : fast_exp2(m_run[nt][h2] - mx);
          if (mv) m_run[nt][h2] = mx;
        }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) o_l[nt][e] *= alpha[nt][e & 1];
#pragma unroll
        for (int m = 0; m < D / 16; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[m][nt][e] *= alpha[nt][e & 1];
      }
    }
    unsigned pk_lo[U][NT], pk_hi[U][NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float r0 = (m_run[nt][0] == -INFINITY) ? 0.f : m_run[nt][0];
      const float r1 = (m_run[nt][1] == -INFINITY) ? 0.f : m_run[nt][1];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        // key quad / quad + 8, heads 2*c4, 2*c4+1
        pk_lo[u][nt] = pack2<FP8 || HALF>(fast_exp2(x[u][nt][0] - r0), fast_exp2(x[u][nt][1] - r1));
        pk_hi[u][nt] = pack2<FP8 || HALF>(fast_exp2(x[u][nt][2] - r0), fast_exp2(x[u][nt][3] - r1));
      }
    }

#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (u >= nu) break;
      const unsigned char* sv = smem + ((i0 + u) % NST) * C::STAGE + C::KV_UNIT;
      // P^T as the B operand (16 keys x 8 heads, "col"): this lane needs head
      // nt*8 + quad at keys 2*c4, 2*c4+1 (b0) and 2*c4+8, 2*c4+9 (b1); they sit
      // in lanes src0 (even key) and src1 (odd key), half quad & 1.
      unsigned pb0[NT], pb1[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const unsigned x0 = __shfl_sync(0xffffffffu, pk_lo[u][nt], src0);
        const unsigned x1 = __shfl_sync(0xffffffffu, pk_lo[u][nt], src1);
        const unsigned y0 = __shfl_sync(0xffffffffu, pk_hi[u][nt], src0);
        const unsigned y1 = __shfl_sync(0xffffffffu, pk_hi[u][nt], src1);
        pb0[nt] = __byte_perm(x0, x1, half_sel);
        pb1[nt] = __byte_perm(y0, y1, half_sel);
      }

      // O^T += V^T P^T: M = d (16 per tile), N = heads, K = the 16 keys.
      if constexpr (FP8) {
        // V^T fragments straight from the e4m3 bytes.  The d axis of V (and so
        // of O) is permuted: tile m, fragment row quad is d = quad*D/8 + 2m and
        // row quad + 8 is d = quad*D/8 + 2m + 1, so each lane reads D/8
        // contiguous bytes of each of its key rows 2*c4, 2*c4+1, 2*c4+8, 2*c4+9.
        unsigned v0[D / 32], v1[D / 32], v2[D / 32], v3[D / 32];
        load_v_bytes<D, HG>(sv, hh, 2 * c4, quad, v0);
        load_v_bytes<D, HG>(sv, hh, 2 * c4 + 1, quad, v1);
        load_v_bytes<D, HG>(sv, hh, 2 * c4 + 8, quad, v2);
        load_v_bytes<D, HG>(sv, hh, 2 * c4 + 9, quad, v3);
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
          // bytes d0 and d0 + 1 of two key rows r, r' interleaved in one
          // word, [r.d0, r'.d0, r.d0+1, r'.d0+1]: its low half is the pair at
          // d0 (fragment row quad), its high half the pair at d0 + 1 (row
          // quad + 8)
          const int wi = m >> 1;
          const unsigned sel = (m & 1) ? 0x7362u : 0x5140u;
          const unsigned x01 = __byte_perm(v0[wi], v1[wi], sel);
          const unsigned x23 = __byte_perm(v2[wi], v3[wi], sel);
          unsigned a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(x01, a0, a1);
          e4m3x4_to_f16x2x2(x23, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816<true>(o[m][nt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
        }
      } else {
        const unsigned sv_a = smem_u32(sv);
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
          unsigned a0, a1, a2, a3;
          ldsm_x4_t(sv_a + raw_off<D, FP8, HG>(hh, v_row, 2 * m + v_csel), a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816<HALF>(o[m][nt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
        }
      }
      // Row sums l = 1^T P^T by the tensor core: every row of the all-ones A
      // tile gives each head's sum of this unit's (rounded) weights.
      constexpr unsigned ONES = (FP8 || HALF) ? 0x3C003C00u : 0x3F803F80u;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_16816<FP8 || HALF>(o_l[nt], ONES, ONES, ONES, ONES, pb0[nt], pb1[nt]);
    }
    // Release the stages once every lane of every consumer warp has read them.
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (u < nu) mbar_arrive(&empty[(i0 + u) % NST]);
    }
  }

#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    l_run[nt][0] = o_l[nt][0];
    l_run[nt][1] = o_l[nt][1];
  }

  // ---------------------------------------------------------------- merge
  // The WPH warps of a KV head saw disjoint units of the partition: the
  // others hand (o, m, l) to warp slot 0 through shared memory (the ring is
  // idle once every consumer has left its loop), in the same fragment layout,
  // and slot 0 merges them with the online-softmax rule.
  if constexpr (WPH > 1) {
    named_bar_sync(1, C::NW * 32);
    float* mb = reinterpret_cast<float*>(smem);
    if (wslot > 0) {
      float* dst = mb + ((wslot - 1) * HG + hh) * C::MERGE_FLOATS * 32 + lane;
      int idx = 0;
#pragma unroll
      for (int m = 0; m < D / 16; ++m)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[32 * idx++] = o[m][nt][e];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          dst[32 * idx++] = m_run[nt][h2];
          dst[32 * idx++] = l_run[nt][h2];
        }
    }
    named_bar_sync(1, C::NW * 32);
    // with a single partition the other slots have nothing left to do
    if (wslot > 0 && S == 1) return;
#pragma unroll
    for (int ws = 1; ws < (wslot == 0 ? WPH : 1); ++ws) {
      const float* src = mb + ((ws - 1) * HG + hh) * C::MERGE_FLOATS * 32 + lane;
      float a_self[NT][2], a_other[NT][2];
      int idx = (D / 16) * NT * 4;
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
      for (int m = 0; m < D / 16; ++m)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o[m][nt][e] = o[m][nt][e] * a_self[nt][e & 1] + src[32 * idx++] * a_other[nt][e & 1];
          }
    }
  }

  // ---------------------------------------------------------------- outputs
  // Slot 0 of each KV head owns its G query heads: normalise and write them
  // (bf16 output) or the partition's (o_p, lse_p) for the merge below.
  const int h0 = g * G;
#pragma unroll
  for (int nt = 0; nt < (wslot == 0 ? NT : 0); ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int head = nt * 8 + 2 * c4 + (e & 1);
      if (head >= G) continue;
      const float L = l_run[nt][e & 1];
      const float M = m_run[nt][e & 1];
      // an unsplit final row includes the head's sink in its normaliser
      const float Ls = (S == 1 && !p.o32) ? L + sink_term(p.sinks, h0 + head, M) : L;
      const float inv = (Ls > 0.f) ? out_scale / Ls : 0.f;
#pragma unroll
      for (int m = 0; m < D / 16; ++m) {
        const int d = FP8 ? (quad * (D / 8) + 2 * m + (e >> 1)) : (16 * m + quad + ((e & 2) ? 8 : 0));
        const float val = o[m][nt][e] * inv;
        if (S == 1) {
          const int64_t oi = (static_cast<int64_t>(t0) * p.H + h0 + head) * D + d;
          if (p.o32) {
            p.o32[oi] = val;
            if (m == 0 && quad == 0 && (e & 2) == 0)
              p.lse32[oi / D] = (L > 0.f) ? M + __log2f(L) : -INFINITY;
          } else if constexpr (HALF)
            static_cast<__half*>(p.out)[oi] = __float2half_rn(val);
          else
            static_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(val);
        } else {
          const int64_t prow = (static_cast<int64_t>(r) * p.H + h0 + head) * S + sp;
          p.o_part[prow * D + d] = val;
          if (m == 0 && quad == 0 && (e & 2) == 0)
            p.lse_part[prow] = (L > 0.f) ? M + __log2f(L) : -INFINITY;
        }
      }
    }

  // ---------------------------------------------------------------- merge of the partitions
  // Each CTA publishes its partition (counts it with a release); the CTA that
  // completes the count of its (request, KV-head group) merges the group's
  // S partitions into the output, so no separate combine launch is needed.
  // All consumer warps are still running; the merging CTA spreads the
  // group's HG * G query heads over them.
  if (S > 1) {
    __shared__ int s_last;
    // The barrier orders every warp's partial stores before thread 0's
    // acquire-release add (a release is cumulative), which publishes them
    // at GPU scope; the add that completes the count acquires every other
    // CTA's, and the second barrier hands that on to this CTA's warps.
    named_bar_sync(2, C::NW * 32);
    if (threadIdx.x == 0) {
      unsigned* cnt = p.counters + static_cast<int64_t>(r) * p.Hkv + grp;
      unsigned prev;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "l"(cnt)
                   : "memory");
      s_last = (prev == static_cast<unsigned>(S - 1)) ? 1 : 0;
      if (s_last) *cnt = 0u;  // every partition of the group has counted
    }
    named_bar_sync(2, C::NW * 32);
    if (!s_last) return;
    // heads in pairs (G is even, or 1: then HG * G = HG and pairs may not fit)
    const int nq = HG * G, h_first = grp * HG * G;
    if (nq % 2 == 0) {
      for (int hq = 2 * warp; hq < nq; hq += 2 * C::NW)
        merge_partitions<D, 2, HALF>(p, r, h_first + hq, t0, lane);
    } else {
      for (int hq = warp; hq < nq; hq += C::NW)
        merge_partitions<D, 1, HALF>(p, r, h_first + hq, t0, lane);
    }
  }
}

template <int D, bool FP8, int NT, int HG, int WPH, bool HALF>
cudaError_t launch_decode_t(const Problem& p, const CUtensorMap& kvmap) {
  using C = DecodeCfg<D, FP8, NT, HG, WPH>;
  auto kern = decode_split_kernel<D, FP8, NT, HG, WPH, HALF>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // e4m3 data is widened to its f16 value; the per-tensor scales go here.
  const float sl2 = p.scale * LOG2E * (FP8 ? p.k_scale : 1.f);
  const float out_scale = FP8 ? p.v_scale : 1.f;
  const long long items = static_cast<long long>(p.B) * (p.Hkv / HG) * p.splits;
  if (items == 0) return cudaSuccess;
  if (p.pdl_launch) {
    // programmatic dependent of the previous kernel in the stream
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(items));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = p.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, kvmap, sl2, out_scale);
  }
  kern<<<static_cast<unsigned>(items), C::THREADS, C::SMEM, p.stream>>>(p, kvmap, sl2, out_scale);
  return cudaGetLastError();
}

// Up to 8 query heads per KV head (one head tile): two warps per KV head
// share each partition; more: one warp per KV head, two head tiles.
template <int D, bool FP8, int HG, bool HALF>
cudaError_t launch_decode_g(const Problem& p, const CUtensorMap& kvmap) {
  return (p.G <= 8) ? launch_decode_t<D, FP8, 1, HG, 2, HALF>(p, kvmap)
                    : launch_decode_t<D, FP8, 2, HG, 1, HALF>(p, kvmap);
}

template <int D, bool FP8, bool HALF>
cudaError_t launch_decode_hg(const Problem& p, const CUtensorMap& kvmap) {
  switch (decode_head_group(p.Hkv, D, FP8)) {
    case 4: return launch_decode_g<D, FP8, 4, HALF>(p, kvmap);
    case 2: return launch_decode_g<D, FP8, 2, HALF>(p, kvmap);
    default: return launch_decode_g<D, FP8, 1, HALF>(p, kvmap);
  }
}

template <int D>
cudaError_t launch_decode_d(const Problem& p, const CUtensorMap& kvmap) {
  if (p.kv_dtype == PATTN_KV_FP8_E4M3) return launch_decode_hg<D, true, false>(p, kvmap);
  if (p.kv_dtype == PATTN_KV_F16) return launch_decode_hg<D, false, true>(p, kvmap);
  return launch_decode_hg<D, false, false>(p, kvmap);
}

}  // namespace

cudaError_t launch_decode(const Problem& p, const CUtensorMap& kvmap) {
  return (p.D == 128) ? launch_decode_d<128>(p, kvmap) : launch_decode_d<64>(p, kvmap);
}

int decode_heads_per_cta(int Hkv, int D, int kv_dtype) {
  return decode_head_group(Hkv, D, kv_dtype == PATTN_KV_FP8_E4M3);
}

}  // namespace pattn
