// prefill.cu -- tcgen05 / TMEM / TMA prefill kernel (sm_103a).
//
// Rows with query_len > 1 (full or chunked prefills) are a dense contraction:
// per 128x128 tile, S = Q K^T and O += P V are two 128x128xD MMAs on the
// 5th-generation tensor cores.  The method is the tiled, IO-aware attention
// of "[vLLM] FlashAttention" (introduction; "paper summary"): Q, K and V tiles
// are staged on chip, the softmax is fused, and the N x N score matrix never
// reaches HBM; the online softmax keeps the result exact (same page, "why this
// design" item 4).
//
// One CTA owns two 128-row query sub-tiles that read the same K/V tiles:
// two query heads of one KV group (GQA, num_queries_per_kv even) or, when the
// group size is odd, two consecutive row tiles of one head.  Twelve warps:
//   warps 0-3  softmax + epilogue of sub-tile A, thread i owns row i (TMEM lane i)
//   warps 4-7  softmax + epilogue of sub-tile B
//   warp  8    TMA producer of both Q tiles (once) and the K tiles, page by
//              page through block_table into a 3-stage ring, one lane per
//              page copy
//   warp  9    MMA issuer (one thread)
//   warp 10    TMA producer of the V tiles (2-stage ring), likewise
//   warp 11    idle (it completes the third warpgroup for setmaxnreg)
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+D), O_B
// [384,384+D).  P (bf16, 64 columns) overwrites the upper half of its S
// buffer and is read back from TMEM as the A operand of P V; the next scores
// of that sub-tile are issued right after P V and overwrite it.  The tensor
// core executes one thread's MMAs in issue order, so P V has read its operand
// before the next S writes the same columns.
//
// The issue order S_A(0), S_B(0), then per key tile j: P V_A(j), S_A(j+1),
// P V_B(j), S_B(j+1) makes the two sub-tiles ping-pong: while one softmax
// warpgroup works on its scores the tensor core runs the other sub-tile's
// MMAs.  Because S_X(j+1) is issued after P V_X(j), the commit that announces
// S_X(j+1) also covers P V_X(j), so a softmax warpgroup may rescale its O in
// TMEM as soon as it sees its next scores.
//
// The cache is addressed by one 4-D TMA tensor map over
// [2 * num_blocks][block_size][num_kv_heads][head_size]; a 128-key tile is
// 128 / block_size page loads (one partial-page load when block_size > 128),
// each landing at its rows' offset of a 128-byte-swizzled tile -- the K-major
// (for S) and MN-major (for P V) operand layouts the MMA descriptors name.
// Pages wholly past seq_len are not loaded; V rows at or past seq_len are
// zeroed in shared memory before P V so stale or NaN slots cannot leak
// through 0 * NaN.  Key tiles wholly outside the causal band or the window are
// never visited; tiles that straddle an edge are masked per element.  The
// running max moves lazily: O is rescaled only when a row max grows by more
// than 2^8, which stays exact because the final normalisation divides by the
// sum taken against the same reference max.
#include "../../include/pattn.h"
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

constexpr int PF_THREADS = 384;
// Register split (setmaxnreg): the two softmax warpgroups take SOFTMAX_REGS
// per thread, the producer / MMA warpgroup gives its share back.  The sum must
// stay within the launch allocation (PF_THREADS x the kernel's register count,
// checked on the host before every launch) or setmaxnreg.inc would wait forever.
constexpr int SOFTMAX_REGS = 216;
constexpr int OTHER_REGS = 72;
constexpr int SPLIT_REGS_TOTAL = 2 * 128 * SOFTMAX_REGS + 128 * OTHER_REGS;
// K and V rings: K gets the extra stage because the next scores need it
// before the next P V needs V.  224 KB of shared memory at head size 128.
constexpr int PF_KST = 3;
constexpr int PF_VST = 2;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
constexpr unsigned FULL = 0xffffffffu;

template <int D>
struct PrefillCfg {
  static constexpr int DH = D / 64;                 // 128-byte column blocks
  static constexpr int HALF = BLOCK_M * 128;        // bytes of one 128-row column block
  static constexpr int TILE = DH * HALF;            // bytes of a Q, K or V tile
  static constexpr int Q_OFF = 0;                   // two Q tiles
  static constexpr int K_OFF = Q_OFF + 2 * TILE;
  static constexpr int V_OFF = K_OFF + PF_KST * TILE;
  static constexpr int BAR_OFF = V_OFF + PF_VST * TILE;
  // + barriers + alignment slack; at least 116 KB so one CTA holds an SM (and
  // its 512 TMEM columns) alone
  static constexpr int SMEM_RAW = BAR_OFF + 512 + 1024;
  static constexpr int SMEM = SMEM_RAW > 118784 ? SMEM_RAW : 118784;
  // TMEM columns of sub-tile X's scores and output
  __device__ static constexpr unsigned s_col(int X) { return X ? 128u : 0u; }
  __device__ static constexpr unsigned o_col(int X) { return X ? 384u : 256u; }
};

struct Bars {
  uint64_t q_full[2];
  uint64_t k_full[PF_KST];
  uint64_t v_full[PF_VST];
  uint64_t k_empty[PF_KST];
  uint64_t v_empty[PF_VST];
  uint64_t s_full[2];   // one phase per key tile of sub-tile X
  uint64_t p_full[2];
  uint64_t o_final[2];  // the last P V of sub-tile X
  uint64_t drain;       // every MMA issued, before TMEM is released
  unsigned tmem_base;
  int abort_flag;
};

struct Sub {
  int h, i0, i_last, x0, x1;
  bool valid;
  __device__ bool active(int kt) const { return valid && kt >= x0 && kt < x1; }
};

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a0, a1) * (b, b) + (c, c) on the paired fp32 pipe.
__device__ __forceinline__ void ffma2(float& a0, float& a1, float b, float c) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%0, %1};\n\t"
      "mov.b64 rb, {%2, %2};\n\t"
      "mov.b64 rc, {%3, %3};\n\t"
      "fma.rn.f32x2 ra, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b), "f"(c));
}

// (s0, s1) += (a0, a1)
__device__ __forceinline__ void fadd2(float& s0, float& s1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rb;\n\t"
      "mov.b64 ra, {%0, %1};\n\t"
      "mov.b64 rb, {%2, %3};\n\t"
      "add.f32x2 ra, ra, rb;\n\t"
      "mov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}

// HALF: q, the cache and out are f16 (else bf16).
template <int D, bool HALF>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_kernel(const Problem p, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kvmap, float sl2) {
  using C = PrefillCfg<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::BAR_OFF);
  unsigned* status = &p.hdr->status;

  // ------------------------------------------------------------ work item
  const bool head_pairs = (p.G % 2) == 0;
  const int NP = head_pairs ? p.H / 2 : p.H;
  const int KC = p.kv_chunks;
  const int chunk = blockIdx.x % KC;
  const int rank = (blockIdx.x / KC) / NP;
  const int pidx = (blockIdx.x / KC) % NP;
  if (rank >= p.hdr->num_prefill_tiles) return;
  const int2 tl = p.tiles[rank];
  const int r = tl.x, qt = tl.y;
  const int t0 = p.qsl[r];
  const int q_len = p.qsl[r + 1] - t0;
  const int s = p.seq_lens[r];
  const int ctx = s - q_len;
  const int W = p.window;

  // Sub-tile X of this item (no array: the softmax warps pick X at run time).
  auto make_sub = [&](int X) {
    Sub u;
    u.h = head_pairs ? 2 * pidx + X : pidx;
    u.i0 = head_pairs ? qt * BLOCK_M : qt * 2 * BLOCK_M + X * BLOCK_M;
    u.valid = u.i0 < q_len;
    u.i_last = min(q_len, u.i0 + BLOCK_M) - 1;
    const int lo = (W > 0) ? max(0, ctx + u.i0 - W + 1) : 0;
    const int hi = p.causal ? min(s, ctx + u.i_last + 1) : s;
    u.x0 = lo / BLOCK_N;
    u.x1 = u.valid ? max(u.x0, (hi + BLOCK_N - 1) / BLOCK_N) : u.x0;
    if (KC > 1) {  // this CTA's chunk of the request's key tiles
      const int per = ((s + BLOCK_N - 1) / BLOCK_N + KC - 1) / KC;
      u.x0 = max(u.x0, chunk * per);
      u.x1 = max(u.x0, min(u.x1, (chunk + 1) * per));
    }
    if (!u.valid) u.x0 = u.x1 = 0;
    return u;
  };
  const Sub subA = make_sub(0), subB = make_sub(1);
  const int u0 = subB.valid ? min(subA.x0, subB.x0) : subA.x0;
  const int u1 = subB.valid ? max(subA.x1, subB.x1) : subA.x1;
  const int n_union = u1 - u0;
  const int g = subA.h / p.G;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], BLOCK_M);
      mbar_init(&bars->o_final[i], 1);
    }
    for (int i = 0; i < PF_KST; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < PF_VST; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
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

  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(OTHER_REGS));
  if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ TMA producers
    // Warp 8 streams Q (once) and the K tiles, warp 10 the V tiles, each
    // through its own ring, so a K tile never queues behind a V slot.  Each
    // warp reads the block ids of a key tile in one coalesced load, one tile
    // ahead.  Lane 0 waits for the stage and posts the tile's bytes; the
    // tile's copies (one per page and d half) then go out from one lane each,
    // so a tile costs one copy instruction, not 2 x pages of them in one
    // thread.
    const int kv = (warp == 10) ? 1 : 0;
    if (n_union > 0) {
      if (kv == 0 && lane == 0) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kvmap);
#pragma unroll
        for (int X = 0; X < 2; ++X) {
          const Sub& u = X ? subB : subA;
          if (!u.valid) continue;
          mbar_arrive_expect_tx(&bars->q_full[X], C::TILE);
#pragma unroll
          for (int dh = 0; dh < C::DH; ++dh)
            tma_load_3d(sQ + X * C::TILE + dh * C::HALF, &qmap, &bars->q_full[X], dh * 64, u.h,
                        t0 + u.i0);
        }
      }
      const int* bt = p.block_table + static_cast<int64_t>(r) * p.bt_stride;
      // block id of page `lane` of key tile kt (0 when that page is past seq_len)
      auto page_block = [&](int kt) {
        const int key0 = kt * BLOCK_N + lane * rows_box;
        int blk = 0;
        if (lane < pages_per_tile && key0 < s) {
          blk = bt[key0 / p.bs];
          if (blk < 0 || blk >= p.NB) {
            flag_status(status, PATTN_DEV_BAD_METADATA);
            blk = min(max(blk, 0), p.NB - 1);
          }
        }
        return blk;
      };
      int blk_next = page_block(u0);
      // Copy `lane` of a tile: page lane / DH, d half lane % DH.
      const int my_pg = lane / C::DH, my_dh = lane % C::DH;
      const int nst = kv ? PF_VST : PF_KST;
      unsigned char* ring = kv ? sV : sK;
      for (int j = 0; j < n_union; ++j) {
        const int key_base = (u0 + j) * BLOCK_N;
        const int my_blk = __shfl_sync(FULL, blk_next, my_pg);
        if (j + 1 < n_union) blk_next = page_block(u0 + j + 1);
        // pages of this tile that hold keys below seq_len
        const int n_load = min(pages_per_tile, (s - key_base + rows_box - 1) / rows_box);
        const int my_key0 = key_base + my_pg * rows_box;
        const int my_slot = p.bs_shift >= 0 ? (my_key0 & (p.bs - 1)) : (my_key0 % p.bs);
        const unsigned bytes = static_cast<unsigned>(n_load * rows_box * 128 * C::DH);
        const int st = j % nst;
        uint64_t* empty = kv ? &bars->v_empty[st] : &bars->k_empty[st];
        uint64_t* full = kv ? &bars->v_full[st] : &bars->k_full[st];
        int ok = 1;
        if (lane == 0) {
          if (j >= nst && !mbar_wait(empty, ((j / nst) - 1) & 1, status, abort_flag))
            ok = 0;
          else
            mbar_arrive_expect_tx(full, bytes);
        }
        if (!__shfl_sync(FULL, ok, 0)) break;
        if (my_pg < n_load)
          tma_load_4d(ring + st * C::TILE + my_dh * C::HALF + my_pg * rows_box * 128, &kvmap, full,
                      my_dh * 64, g, my_slot, kv * p.NB + my_blk);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_union > 0) {
      constexpr unsigned idesc_s = make_idesc_f16(BLOCK_M, BLOCK_N, !HALF, false);
      constexpr unsigned idesc_pv = make_idesc_f16(BLOCK_M, D, !HALF, true);
      // Base descriptors; a byte offset o moves the start address field by
      // o >> 4 (shared addresses stay far below the field's 256 KB range).
      const uint64_t q_d = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t k_d = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t v_d = smem_desc_sw128(smem_u32(sV), C::HALF, 1024);
      int n_pv0 = 0, n_pv1 = 0;
      bool q_ready0 = false, q_ready1 = false;
      bool ok = true;
      for (int j = 0; ok && j <= n_union; ++j) {
        const int kt = u0 + j;
        bool k_ready = false, v_ready = false;
        // Unrolled: every per-sub-tile value stays in a register (a runtime
        // choice between two locals would put them in local memory).
#pragma unroll
        for (int X = 0; X < 2; ++X) {
          const Sub& u = X ? subB : subA;
          int& n_pv = X ? n_pv1 : n_pv0;
          bool& q_ready = X ? q_ready1 : q_ready0;
          // P V for the previous key tile
          if (j >= 1 && u.active(kt - 1)) {
            const int stp = (j - 1) % PF_VST;
            if (!mbar_wait(&bars->p_full[X], n_pv & 1, status, abort_flag)) {
              ok = false;
              break;
            }
            if (!v_ready) {
              if (!mbar_wait(&bars->v_full[stp], ((j - 1) / PF_VST) & 1, status, abort_flag)) {
                ok = false;
                break;
              }
              v_ready = true;
            }
            tc_fence_after();
            const unsigned p_t = tmem + C::s_col(X) + 64;
            const unsigned o_t = tmem + C::o_col(X);
            const uint64_t vb = v_d + ((stp * C::TILE) >> 4);
#pragma unroll
            for (int kk = 0; kk < BLOCK_N / 16; ++kk)
              tc_mma_ts(o_t, p_t + kk * 8, vb + ((kk * 16 * 128) >> 4), idesc_pv,
                        (n_pv > 0 || kk > 0) ? 1u : 0u);
            ++n_pv;
            if (kt - 1 == u.x1 - 1) tc_commit(&bars->o_final[X]);
            if (X == 1 || !subB.active(kt - 1)) tc_commit(&bars->v_empty[stp]);
          }
          // scores for this key tile
          if (j < n_union && u.active(kt)) {
            const int st = j % PF_KST;
            if (!k_ready) {
              if (!mbar_wait(&bars->k_full[st], (j / PF_KST) & 1, status, abort_flag)) {
                ok = false;
                break;
              }
              k_ready = true;
            }
            if (!q_ready) {
              if (!mbar_wait(&bars->q_full[X], 0, status, abort_flag)) {
                ok = false;
                break;
              }
              q_ready = true;
            }
            tc_fence_after();
            const uint64_t qb = q_d + ((X * C::TILE) >> 4);
            const uint64_t kb = k_d + ((st * C::TILE) >> 4);
            const unsigned s_t = tmem + C::s_col(X);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const unsigned off = ((kk >> 2) * C::HALF + (kk & 3) * 32) >> 4;
              tc_mma_ss(s_t, qb + off, kb + off, idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(&bars->s_full[X]);
            if (X == 1 || !subB.active(kt)) tc_commit(&bars->k_empty[st]);
          }
        }
      }
      // No MMA may still be running when TMEM is released (matters only when
      // a role gave up on a wait).
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, status, nullptr);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(SOFTMAX_REGS));
    // ------------------------------------------------------------ softmax warpgroups
    const int X = warp >> 2;            // 0: A (warps 0-3), 1: B (warps 4-7)
    const Sub u = make_sub(X);
    const int row = threadIdx.x & 127;  // TMEM lane
    const int i = u.i0 + row;
    const int pos = ctx + i;
    const int kmax_row = p.causal ? min(s, pos + 1) : s;
    const unsigned lane_base = tmem + (static_cast<unsigned>((warp & 3) * 32) << 16);
    const unsigned s_t = lane_base + C::s_col(X);
    const unsigned o_t = lane_base + C::o_col(X);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = u.valid;
    const int nt = u.x1 - u.x0;
    for (int c = 0; ok && c < nt; ++c) {
      const int kt = u.x0 + c;
      const int key0 = kt * BLOCK_N;
      if (!__all_sync(FULL, mbar_wait(&bars->s_full[X], c & 1, status, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[BLOCK_N];
#pragma unroll
      for (int q = 0; q < BLOCK_N / 32; ++q)
        tc_ld32(s_t + q * 32, *reinterpret_cast<float(*)[32]>(&sv[q * 32]));
      tc_wait_ld();

      // Does any row of this sub-tile see a masked key in this tile?
      const bool edge = (key0 + BLOCK_N > s) ||
                        (p.causal && key0 + BLOCK_N - 1 > ctx + u.i0) ||
                        (W > 0 && (ctx + u.i_last) - key0 >= W);
      if (edge) {
        // column limits of this row in the tile: visible iff lim_lo <= q < lim_hi
        const int lim_hi = kmax_row - key0;
        const int lim_lo = (W > 0) ? pos - W + 1 - key0 : -1;
#pragma unroll
        for (int q = 0; q < BLOCK_N; ++q)
          sv[q] = (q < lim_hi && q >= lim_lo) ? sv[q] : -INFINITY;
      }
      float m4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
      for (int q = 4; q < BLOCK_N - 4; q += 8) {
        m4[0] = max3(m4[0], sv[q + 0], sv[q + 1]);
        m4[1] = max3(m4[1], sv[q + 2], sv[q + 3]);
        m4[2] = max3(m4[2], sv[q + 4], sv[q + 5]);
        m4[3] = max3(m4[3], sv[q + 6], sv[q + 7]);
      }
      m4[0] = max3(m4[0], sv[BLOCK_N - 4], sv[BLOCK_N - 3]);
      m4[1] = max3(m4[1], sv[BLOCK_N - 2], sv[BLOCK_N - 1]);
      const float mx = max3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
      const float mx_s = (mx == -INFINITY) ? -INFINITY : mx * sl2;

      // Lazy rescale: move the reference max only when it grows by > 2^8.
      const bool grow = mx_s > m_run + RESCALE_THRESHOLD;
      const bool need_o = grow && (m_run != -INFINITY) && (c > 0);
      float alpha = 1.f;
      if (grow) {
        alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - mx_s);
        l_run *= alpha;
        m_run = mx_s;
      }
      if (__any_sync(FULL, need_o)) {
        // P V of the previous tile is complete: the commit that announced
        // these scores was issued after it.
        const float a = need_o ? alpha : 1.f;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          float ov[32];
          tc_ld32(o_t + q * 32, ov);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] *= a;
          tc_st32(o_t + q * 32, ov);
        }
      }

      const float neg_m = -((m_run == -INFINITY) ? 0.f : m_run);
      float ps0 = 0.f, ps1 = 0.f, ps2 = 0.f, ps3 = 0.f;
#pragma unroll
      for (int q = 0; q < BLOCK_N; q += 32) {
        unsigned pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          float a0 = sv[q + e], a1 = sv[q + e + 1], a2 = sv[q + e + 2], a3 = sv[q + e + 3];
          ffma2(a0, a1, sl2, neg_m);
          ffma2(a2, a3, sl2, neg_m);
          a0 = fast_exp2(a0);
          a1 = fast_exp2(a1);
          a2 = fast_exp2(a2);
          a3 = fast_exp2(a3);
          fadd2(ps0, ps1, a0, a1);
          fadd2(ps2, ps3, a2, a3);
          pk[e / 2] = pack2<HALF>(a0, a1);
          pk[e / 2 + 1] = pack2<HALF>(a2, a3);
        }
        tc_st16u(s_t + 64 + q / 2, pk);
      }
      l_run += (ps0 + ps1) + (ps2 + ps3);
      tc_wait_st();

      // Zero V rows at or past seq_len before P V reads them (done by the
      // first sub-tile whose P V reads this tile).
      if (key0 + BLOCK_N > s && (X == 0 || !subA.active(kt))) {
        const int j = kt - u0;
        const int st = j % PF_VST;
        if (!__all_sync(FULL, mbar_wait(&bars->v_full[st], (j / PF_VST) & 1, status, abort_flag))) {
          ok = false;
          break;
        }
        if (key0 + row >= s) {
          unsigned char* vrow = sV + st * C::TILE + row * 128;
#pragma unroll
          for (int dh = 0; dh < C::DH; ++dh)
#pragma unroll
            for (int b = 0; b < 128; b += 16)
              *reinterpret_cast<uint4*>(vrow + dh * C::HALF + b) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&bars->p_full[X]);
    }

    // ------------------------------------------------------------ epilogue
    // The normalised row goes to out, or (partial-result mode) to o32 in
    // fp32 with its log2-domain lse = m + log2(l).
    const int64_t ri = (static_cast<int64_t>(t0 + i) * p.H + u.h) * KC + chunk;  // o32 / lse32 row
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                          (static_cast<int64_t>(t0 + i) * p.H + u.h) * D;
    if (u.valid && ok && nt > 0 &&
        __all_sync(FULL, mbar_wait(&bars->o_final[X], 0, status, abort_flag))) {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll
      for (int q = 0; q < D / 32; ++q) {
        float ov[32];
        tc_ld32(o_t + q * 32, ov);
        tc_wait_ld();
        if (i < q_len) {
          if (p.o32) {
            float4* dst = reinterpret_cast<float4*>(p.o32 + ri * D + q * 32);
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              dst[e / 4] = make_float4(ov[e] * inv, ov[e + 1] * inv, ov[e + 2] * inv, ov[e + 3] * inv);
          } else {
            unsigned pkd[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pkd[e] = pack2<HALF>(ov[2 * e] * inv, ov[2 * e + 1] * inv);
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              *reinterpret_cast<uint4*>(orow + q * 32 + e * 2) =
                  make_uint4(pkd[e], pkd[e + 1], pkd[e + 2], pkd[e + 3]);
          }
        }
      }
      if (p.o32 && i < q_len) p.lse32[ri] = (l_run > 0.f) ? m_run + __log2f(l_run) : -INFINITY;
    } else if (u.valid && i < q_len) {
      if (p.o32) {
        for (int e = 0; e < D; ++e) p.o32[ri * D + e] = 0.f;
        p.lse32[ri] = -INFINITY;
      } else {
        for (int e = 0; e < D; ++e) orow[e] = __float2bfloat16_rn(0.f);
      }
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

int prefill_rows_per_item(int G) { return (G % 2 == 0) ? BLOCK_M : 2 * BLOCK_M; }

template <int D, bool HALF>
cudaError_t launch_prefill_t(const Problem& p, const CUtensorMap& q_map, const CUtensorMap& kv_map,
                             unsigned grid) {
  auto k = prefill_kernel<D, HALF>;
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, k);
  if (e != cudaSuccess) return e;
  // The register split must fit in what the CTA is launched with.
  if (static_cast<long long>(attr.numRegs) * PF_THREADS < SPLIT_REGS_TOTAL)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, PrefillCfg<D>::SMEM);
  if (e != cudaSuccess) return e;
  // Scores are scaled to log2 units by sl2 = scale * log2(e).  It is kept
  // strictly positive so a masked score (-inf) always maps to exp2(-inf) = 0;
  // at scale == 0 the visible scores become ~1e-30 * q.k, whose exp2 is 1.0f
  // exactly (uniform weights, as the definition gives).
  const float sl2 = fmaxf(p.scale * LOG2E, 1e-30f);
  k<<<grid, PF_THREADS, PrefillCfg<D>::SMEM, p.stream>>>(p, q_map, kv_map, sl2);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const Problem& p, const CUtensorMap& q_map, const CUtensorMap& kv_map) {
  const int NP = (p.G % 2 == 0) ? p.H / 2 : p.H;
  const long long grid = static_cast<long long>(p.max_tiles) * NP * p.kv_chunks;
  if (grid == 0) return cudaSuccess;
  const unsigned g = static_cast<unsigned>(grid);
  if (p.kv_dtype == PATTN_KV_F16)
    return p.D == 128 ? launch_prefill_t<128, true>(p, q_map, kv_map, g)
                      : launch_prefill_t<64, true>(p, q_map, kv_map, g);
  return p.D == 128 ? launch_prefill_t<128, false>(p, q_map, kv_map, g)
                    : launch_prefill_t<64, false>(p, q_map, kv_map, g);
}

}  // namespace pattn
