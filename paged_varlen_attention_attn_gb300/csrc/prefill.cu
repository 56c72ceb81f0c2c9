// prefill.cu -- tcgen05 / TMEM / TMA prefill kernel (sm_103a).
//
// Rows with query_len > 1 (full or chunked prefills) are a dense contraction:
// per 128x128 tile, S = Q K^T and O += P V are two 128x128xD MMAs on the
// 5th-generation tensor cores.  The method is the tiled, IO-aware attention
// of "[vLLM] FlashAttention" (introduction; "paper summary"): Q, K and V tiles
// are staged in on-chip memory, the softmax is fused, and the N x N score
// matrix never reaches HBM; the online softmax keeps the result exact (same
// page, "why this design" item 4).
//
// One CTA computes one 128-row query tile of one head (rows of one request),
// six warps:
//   warps 0-3  softmax + epilogue, thread i owns query row i (TMEM lane i);
//   warp  4    TMA producer: the Q tile once, then K and V tiles page by page
//              through block_table into a NST-stage ring;
//   warp  5    MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//              score buffers, then O += P_j V_j with P_j read back from TMEM.
// TMEM: S buffers at columns [0,128) and [128,256), O at [256, 256 + D).
// P_j (bf16) overwrites the first 64 columns of its own S buffer.
//
// The cache is addressed by one 4-D TMA tensor map over
// [2 * num_blocks][block_size][num_kv_heads][head_size]; a 128-key tile is
// 128 / block_size page loads (or one partial-page load when block_size >
// 128), each landing at its rows' offset of a 128-byte-swizzled tile, which is
// exactly the K-major (for S) and MN-major (for P V) operand layout the MMA
// descriptors name.  Pages wholly past seq_len are not loaded; V rows at or
// past seq_len are zeroed in shared memory before P V so stale or NaN slots
// cannot leak through 0 * NaN.
//
// Key tiles wholly outside the causal band or the window are never visited;
// tiles that straddle an edge are masked per element.  The running max is
// updated lazily: O in TMEM is rescaled only when a row max grows by more
// than 2^8, which keeps the result exact because the final normalisation
// divides by the sum taken with the same reference max.
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

constexpr int PF_THREADS = 192;
constexpr int PF_NST = 2;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

template <int D>
struct PrefillCfg {
  static constexpr int DH = D / 64;                 // 128-byte column blocks
  static constexpr int HALF = BLOCK_M * 128;        // bytes of one 128-row column block
  static constexpr int TILE = DH * HALF;            // bytes of a Q, K or V tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE;
  static constexpr int V_OFF = K_OFF + PF_NST * TILE;
  static constexpr int BAR_OFF = V_OFF + PF_NST * TILE;
  // + barriers + alignment slack; at least 116 KB so one CTA holds an SM
  // (and its 512 TMEM columns) alone
  static constexpr int SMEM_RAW = BAR_OFF + 256 + 1024;
  static constexpr int SMEM = SMEM_RAW > 118784 ? SMEM_RAW : 118784;
  static constexpr unsigned S_COL0 = 0, S_COL1 = 128, O_COL = 256;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[PF_NST];
  uint64_t v_full[PF_NST];
  uint64_t kv_empty[PF_NST];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done;   // one phase per P V
  uint64_t o_final;  // the last P V only (an unambiguous wait for the epilogue)
  uint64_t drain;    // every MMA issued, before TMEM is released
  unsigned tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_kernel(const Problem p, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kvmap, float sl2) {
  using C = PrefillCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::BAR_OFF);
  unsigned* status = &p.hdr->status;

  const int rank = blockIdx.x / p.H;
  const int h = blockIdx.x % p.H;
  if (rank >= p.hdr->num_prefill_tiles) return;
  const int2 tl = p.tiles[rank];
  const int r = tl.x, qt = tl.y;
  const int t0 = p.qsl[r];
  const int q_len = p.qsl[r + 1] - t0;
  const int s = p.seq_lens[r];
  const int ctx = s - q_len;
  const int i0 = qt * BLOCK_M;
  const int i_last = min(q_len, i0 + BLOCK_M) - 1;
  const int g = h / p.G;
  const int W = p.window;
  const int lo = (W > 0) ? max(0, ctx + i0 - W + 1) : 0;
  const int hi = p.causal ? min(s, ctx + i_last + 1) : s;
  const int kt_begin = lo / BLOCK_N;
  const int n_tiles = max(0, (hi + BLOCK_N - 1) / BLOCK_N - kt_begin);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < PF_NST; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], BLOCK_M);
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_final, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const unsigned tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;

  unsigned char* sQ = smem + C::Q_OFF;
  unsigned char* sK = smem + C::K_OFF;
  unsigned char* sV = smem + C::V_OFF;
  const int rows_box = p.bs < BLOCK_N ? p.bs : BLOCK_N;
  const int pages_per_tile = BLOCK_N / rows_box;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kvmap);
      mbar_arrive_expect_tx(&bars->q_full, C::TILE);
#pragma unroll
      for (int dh = 0; dh < C::DH; ++dh)
        tma_load_3d(sQ + dh * C::HALF, &qmap, &bars->q_full, dh * 64, h, t0 + i0);
      const int* bt = p.block_table + static_cast<int64_t>(r) * p.mbps;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % PF_NST;
        if (j >= PF_NST && !mbar_wait(&bars->kv_empty[st], ((j / PF_NST) - 1) & 1, status, abort_flag))
          break;
        const int key_base = (kt_begin + j) * BLOCK_N;
        int n_load = 0;
        for (int pg = 0; pg < pages_per_tile; ++pg)
          if (key_base + pg * rows_box < s) ++n_load;
        const unsigned bytes = static_cast<unsigned>(n_load * rows_box * 128 * C::DH);
        unsigned char* dk = sK + st * C::TILE;
        unsigned char* dv = sV + st * C::TILE;
        mbar_arrive_expect_tx(&bars->k_full[st], bytes);
        mbar_arrive_expect_tx(&bars->v_full[st], bytes);
        for (int pg = 0; pg < pages_per_tile; ++pg) {
          const int key0 = key_base + pg * rows_box;
          if (key0 >= s) break;
          int blk = bt[key0 / p.bs];
          if (blk < 0 || blk >= p.NB) {
            flag_status(status, PATTN_DEV_BAD_METADATA);
            blk = min(max(blk, 0), p.NB - 1);
          }
          const int slot = key0 % p.bs;
#pragma unroll
          for (int dh = 0; dh < C::DH; ++dh) {
            tma_load_4d(dk + dh * C::HALF + pg * rows_box * 128, &kvmap, &bars->k_full[st],
                        dh * 64, g, slot, blk);
            tma_load_4d(dv + dh * C::HALF + pg * rows_box * 128, &kvmap, &bars->v_full[st],
                        dh * 64, g, slot, p.NB + blk);
          }
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr unsigned idesc_s = make_idesc_f16(BLOCK_M, BLOCK_N, true, false);
      constexpr unsigned idesc_pv = make_idesc_f16(BLOCK_M, D, true, true);
      const unsigned q_a = smem_u32(sQ), k_a = smem_u32(sK), v_a = smem_u32(sV);
      auto issue_s = [&](int j) {
        const int st = j % PF_NST;
        const unsigned d_t = tmem + ((j & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const unsigned off = (kk >> 2) * C::HALF + (kk & 3) * 32;
          const uint64_t ad = smem_desc_sw128(q_a + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(k_a + st * C::TILE + off, 16, 1024);
          tc_mma_ss(d_t, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&bars->s_full[j & 1]);
      };
      bool ok = mbar_wait(&bars->q_full, 0, status, abort_flag);
      if (ok) ok = mbar_wait(&bars->k_full[0], 0, status, abort_flag);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
          const int st1 = (j + 1) % PF_NST;
          if (!mbar_wait(&bars->k_full[st1], ((j + 1) / PF_NST) & 1, status, abort_flag)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        const int st = j % PF_NST;
        if (!mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1, status, abort_flag)) break;
        if (!mbar_wait(&bars->v_full[st], (j / PF_NST) & 1, status, abort_flag)) break;
        tc_fence_after();
        const unsigned p_t = tmem + ((j & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
        for (int kk = 0; kk < BLOCK_N / 16; ++kk) {
          const uint64_t bd =
              smem_desc_sw128(v_a + st * C::TILE + kk * 16 * 128, C::HALF, 1024);
          tc_mma_ts(tmem + C::O_COL, p_t + kk * 8, bd, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&bars->o_done);
        tc_commit(&bars->kv_empty[st]);
        if (j == n_tiles - 1) tc_commit(&bars->o_final);
      }
      // No MMA may still be running when TMEM is released (matters only when
      // a role gave up on a wait).
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, status, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int row = threadIdx.x;  // 0..127 == TMEM lane
    const int i = i0 + row;
    const int pos = ctx + i;
    const int kmax_row = p.causal ? min(s, pos + 1) : s;
    const int kmin_row = (W > 0) ? pos - W + 1 : -0x7fffffff;
    const unsigned lane_addr = tmem + (static_cast<unsigned>(warp * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int kt = kt_begin + j;
      const int key0 = kt * BLOCK_N;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[j & 1], (j >> 1) & 1, status, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const unsigned s_t = lane_addr + ((j & 1) ? C::S_COL1 : C::S_COL0);
      float sv[BLOCK_N];
#pragma unroll
      for (int c = 0; c < BLOCK_N / 32; ++c)
        tc_ld32(s_t + c * 32, *reinterpret_cast<float(*)[32]>(&sv[c * 32]));
      tc_wait_ld();

      // Does any row of this tile see a masked key in it?
      const bool edge = (key0 + BLOCK_N > s) || (p.causal && key0 + BLOCK_N - 1 > ctx + i0) ||
                        (W > 0 && (ctx + i_last) - key0 >= W);
      float mx = -INFINITY;
      if (edge) {
#pragma unroll
        for (int c = 0; c < BLOCK_N; ++c) {
          const int k = key0 + c;
          const bool vis = (k < kmax_row) && (k >= kmin_row);
          sv[c] = vis ? sv[c] : -INFINITY;
          mx = fmaxf(mx, sv[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < BLOCK_N; ++c) mx = fmaxf(mx, sv[c]);
      }
      const float mx_s = (mx == -INFINITY) ? -INFINITY : mx * sl2;

      // Lazy rescale: move the reference max only when it grows by > 2^8.
      const bool grow = mx_s > m_run + RESCALE_THRESHOLD;
      const bool need_o = grow && (m_run != -INFINITY) && (j > 0);
      float alpha = 1.f;
      if (grow) {
        alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - mx_s);
        l_run *= alpha;
        m_run = mx_s;
      }
      if (__any_sync(0xffffffffu, need_o)) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->o_done, (j - 1) & 1, status, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float a = need_o ? alpha : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tc_ld32(lane_addr + C::O_COL + c * 32, ov);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] *= a;
          tc_st32(lane_addr + C::O_COL + c * 32, ov);
        }
      }

      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      float psum = 0.f;
      unsigned pk[BLOCK_N / 2];
#pragma unroll
      for (int c = 0; c < BLOCK_N; c += 2) {
        float p0 = fast_exp2(fmaf(sv[c], sl2, -m_use));
        float p1 = fast_exp2(fmaf(sv[c + 1], sl2, -m_use));
        if (edge) {
          p0 = (sv[c] == -INFINITY) ? 0.f : p0;
          p1 = (sv[c + 1] == -INFINITY) ? 0.f : p1;
        }
        psum += p0 + p1;
        pk[c / 2] = pack2<false>(p0, p1);
      }
      l_run += psum;
#pragma unroll
      for (int c = 0; c < BLOCK_N / 2; c += 16)
        tc_st16u(s_t + c, *reinterpret_cast<unsigned(*)[16]>(&pk[c]));
      tc_wait_st();

      // Zero V rows at or past seq_len before P V reads them.
      if (key0 + BLOCK_N > s) {
        const int st = j % PF_NST;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (j / PF_NST) & 1, status, abort_flag))) {
          ok = false;
          break;
        }
        if (key0 + row >= s) {
          unsigned char* vrow = sV + st * C::TILE + row * 128;
#pragma unroll
          for (int dh = 0; dh < C::DH; ++dh)
#pragma unroll
            for (int c = 0; c < 128; c += 16)
              *reinterpret_cast<uint4*>(vrow + dh * C::HALF + c) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&bars->p_full[j & 1]);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n_tiles > 0 &&
        __all_sync(0xffffffffu, mbar_wait(&bars->o_final, 0, status, abort_flag))) {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                            (static_cast<int64_t>(t0 + i) * p.H + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tc_ld32(lane_addr + C::O_COL + c * 32, ov);
        tc_wait_ld();
        if (i < q_len) {
          unsigned pkd[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) pkd[e] = pack2<false>(ov[2 * e] * inv, ov[2 * e + 1] * inv);
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<uint4*>(orow + c * 32 + e * 2) =
                make_uint4(pkd[e], pkd[e + 1], pkd[e + 2], pkd[e + 3]);
        }
      }
    } else if (i < q_len) {
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                            (static_cast<int64_t>(t0 + i) * p.H + h) * D;
      for (int c = 0; c < D; ++c) orow[c] = __float2bfloat16_rn(0.f);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_prefill(const Problem& p, const CUtensorMap& q_map, const CUtensorMap& kv_map) {
  const long long grid = static_cast<long long>(p.max_tiles) * p.H;
  if (grid == 0) return cudaSuccess;
  const float sl2 = p.scale * LOG2E;
  if (p.D == 128) {
    auto k = prefill_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PrefillCfg<128>::SMEM);
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(grid), PF_THREADS, PrefillCfg<128>::SMEM, p.stream>>>(p, q_map, kv_map, sl2);
  } else {
    auto k = prefill_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PrefillCfg<64>::SMEM);
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(grid), PF_THREADS, PrefillCfg<64>::SMEM, p.stream>>>(p, q_map, kv_map, sl2);
  }
  return cudaGetLastError();
}

}  // namespace pattn
