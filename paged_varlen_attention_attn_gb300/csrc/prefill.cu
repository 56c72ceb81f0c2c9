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
// A work item is two 128-row query sub-tiles that read the same K/V tiles:
// two query heads of one KV group (GQA, num_queries_per_kv even) or, when the
// group size is odd, two consecutive row tiles of one head.  The kernel is
// persistent: one CTA per SM walks a fixed sequence of items from the
// longest-first list, so one item's loads and first scores overlap the end of
// the previous one instead of a CTA launch, set-up and drain.  Twelve warps:
//   warps 0-3  softmax + epilogue of sub-tile A, thread i owns row i (TMEM lane i)
//              (over an e4m3 cache they also split (d 128) or convert (d 64)
//              their Q tile, below)
//   warps 4-7  softmax + epilogue of sub-tile B, likewise
//   warp  8    TMA producer of both Q tiles of each item and the K tiles, page by
//              page through block_table into a 3-stage ring, one lane per
//              page copy (over an e4m3 cache it also widens each K tile at d
//              64, and rows 80-127 of each V tile at d 128)
//   warp  9    MMA issuer (one thread): sub-tile A's MMAs (both sub-tiles'
//              over an e4m3 cache at d 64)
//   warp 10    TMA producer of the V tiles (2-stage ring; 3 over an e4m3 cache
//              at d 128), one page per copy (over an e4m3 cache it also widens
//              each V tile to f16, rows 0-79 of it at d 128)
//   warp 11    MMA issuer of sub-tile B (the two issuers take turns); idle
//              over an e4m3 cache at d 64
// Over an e4m3 cache at d 128 the scores are 8-bit MMAs (kind::f8f6f4) on the
// cache's K codes as TMA lands them: each softmax thread splits its bf16 Q row,
// scaled by a power of two, into e4m3 hi and lo codes whose sum is the scaled
// row, and S is hi K^T + lo K^T in fp32 (exact products), scaled back in the
// softmax.  P V stays an f16 MMA on widened V tiles.
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+D), O_B
// [384,384+D).  P (bf16, 64 columns) overwrites the lower half of its S
// buffer and is read back from TMEM as the A operand of P V; the next scores
// of that sub-tile are issued right after P V, by the same thread, and
// overwrite it.  The tensor core executes one thread's MMAs in issue order,
// so P V has read its operand before the next S writes the same columns.
//
// The issue order S_A(0), S_B(0), then per key tile j: P V_A(j), S_A(j+1),
// P V_B(j), S_B(j+1) makes the two sub-tiles ping-pong: while one softmax
// warpgroup works on its scores the tensor core runs the other sub-tile's
// MMAs.  Because S_X(j+1) is issued after P V_X(j), the commit that announces
// S_X(j+1) also covers P V_X(j), so a softmax warpgroup may rescale its O in
// TMEM as soon as it sees its next scores.
//
// The cache is addressed through TMA tensor maps over
// [2 * num_blocks][block_size][num_kv_heads][head_size].  A K tile is
// 128 / block_size page loads per d half (one partial-page load when
// block_size > 128), each landing at its rows' offset of a 128-byte-swizzled
// column block (the K-major operand of S); a V tile is one load per page, of
// both d halves, landing as 16-key groups (the MN-major operand of P V).
// Pages wholly past seq_len are not loaded; V rows at or past seq_len are
// zeroed in shared memory before P V so stale or NaN slots cannot leak
// through 0 * NaN.  Key tiles wholly outside the causal band or the window are
// never visited; tiles that straddle an edge are masked per element.  The
// running max moves lazily: O is rescaled only when a row max grows by more
// than 2^8, which stays exact because the final normalisation divides by the
// sum taken against the same reference max.
#include <algorithm>

#include "../../include/pattn.h"
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

constexpr int PF_THREADS = 384;
// Register split (setmaxnreg): the two softmax warpgroups take
// softmax_regs(FP8) per thread, the producer / MMA warpgroup gives its share
// back (other_regs).  An e4m3 call's producer widens tiles and needs more.
// The sum must stay within the launch allocation (PF_THREADS x the kernel's
// register count, checked on the host before every launch) or
// setmaxnreg.inc would wait forever; both splits total SPLIT_REGS_TOTAL.
__host__ __device__ constexpr int softmax_regs(bool fp8) { return fp8 ? 200 : 216; }
__host__ __device__ constexpr int other_regs(bool fp8) { return fp8 ? 104 : 72; }
constexpr int SPLIT_REGS_TOTAL = 2 * 128 * softmax_regs(false) + 128 * other_regs(false);
static_assert(2 * 128 * softmax_regs(true) + 128 * other_regs(true) == SPLIT_REGS_TOTAL,
              "both register splits fit the same launch allocation");
// K and V rings: K gets the extra stage because the next scores need it
// before the next P V needs V.  224 KB of shared memory at head size 128.
// Over an e4m3 cache at d 128 a K stage holds the 16 KB of codes only, and
// the space saved gives V (widened in place, after its copy lands) a third
// stage, so its copies run two tiles ahead of the widening.
constexpr int PF_KST = 3;
constexpr int PF_VST = 2;
constexpr int PF_VST_MAX = 3;
// Item ring: the indices of this CTA's next items, claimed one ahead by warp 8
constexpr int PF_RING = 4;
// Rounds of the item list at its end that CTAs claim as they get free
constexpr int DYN_ROUNDS = 4;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
// 2^RESCALE_THRESHOLD: if any of a row's weights against an unmoved
// reference exceeds it, so does their sum; a sum above this sends the tile
// down the path that takes the row max (a larger sum with every weight in
// range only costs that path).
constexpr float FAST_SUM_LIMIT = 256.0f;
constexpr unsigned FULL = 0xffffffffu;

// A 16-bit V tile sits in shared memory as groups of 16 keys, each group's d
// halves one after the other ([key / 16][d half][key % 16][128 bytes]), so
// that one copy moves a whole page; an e4m3 V tile is widened into the K tile
// layout ([d half][key][128 bytes]), the same with groups of V_ROWS = BLOCK_N.
template <bool FP8>
__host__ __device__ constexpr int v_rows() { return FP8 ? BLOCK_N : 16; }

// NK: e4m3 K codes used as they are (an e4m3 cache at d 128).
template <int D, bool NK = false>
struct PrefillCfg {
  static constexpr int DH = D / 64;                 // 128-byte column blocks
  static constexpr int HALF = BLOCK_M * 128;        // bytes of one 128-row column block
  static constexpr int TILE = DH * HALF;            // bytes of a Q, K or V tile
  static constexpr int KSTAGE = NK ? BLOCK_N * D : TILE;  // bytes of a K ring stage
  static constexpr int VST = NK ? PF_VST_MAX : PF_VST;    // V ring stages
  // An e4m3 K or V tile (rows of D bytes) lands at the top of its ring stage
  // and is widened there, in place, to the f16 tile.
  static constexpr int SRC8 = TILE - BLOCK_N * D;
  static constexpr int Q_OFF = 0;                   // two Q tiles
  static constexpr int K_OFF = Q_OFF + 2 * TILE;
  static constexpr int V_OFF = K_OFF + PF_KST * KSTAGE;
  static constexpr int BAR_OFF = V_OFF + VST * TILE;
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
  uint64_t v_full[PF_VST_MAX];
  uint64_t k_empty[PF_KST];
  uint64_t v_empty[PF_VST_MAX];
  uint64_t s_full[2];   // one phase per key tile of sub-tile X
  uint64_t k_land[PF_KST];  // e4m3 K tile landed at the top of its stage (FP8)
  uint64_t v_land[PF_VST_MAX];  // e4m3 V tile landed at the top of its stage (FP8)
  uint64_t q_conv[2];   // Q tile of sub-tile X converted to f16 by its warpgroup (FP8)
  uint64_t p_full[2];
  uint64_t o_final[2];  // the last P V of sub-tile X
  uint64_t q_empty;     // every S MMA of an item issued and done: Q may be replaced
  uint64_t drain;       // every MMA issued, before TMEM is released
  uint64_t tok[2];      // issuer X may take its turn (two MMA issuers)
  uint64_t ring_full[PF_RING];   // slot i holds the index of this CTA's next item
  uint64_t ring_empty[PF_RING];  // every role has taken slot i
  int ring[PF_RING];
  unsigned tmem_base;
  int abort_flag;
};

static_assert(sizeof(Bars) <= 512, "the barriers fit the space kept for them");

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

// Widens rows [row0, row1) of an e4m3 tile, stored as rows of D bytes
// in the last BLOCK_N x D bytes of a K or V stage, in place into the stage's
// f16 tile in the 128-byte-swizzled layout: code c of row r goes to d half
// c / 64, 16-byte chunk (c % 64) / 8, which sits at chunk position
// (chunk ^ (r % 8)) of the row.  A lane takes 16 codes (a piece) per pass,
// and a pass of the warp covers 512 source bytes (512 / D rows); the lane
// keeps the same row offset r0 and piece c in every pass.  At d 128 the two
// rows of a quarter-warp take opposite d halves, so its 16-byte loads and
// stores each land on eight distinct bank groups.  A batch of U passes loads
// all its pieces before any store: f16 rows overlap only source rows at or
// below the batch's last row (at d 128 the second d half of row r is
// exactly source row r; at d 64 f16 row r >= 64 covers source rows 2r - 128
// and 2r - 127), so every source row is read before it is overwritten.  row0
// and row1 are multiples of 16, so passes come in whole batches.  At d 128,
// where f16 row r overlaps source row r alone, warps may widen disjoint row
// ranges of one tile at the same time.
template <int D>
__device__ __forceinline__ void widen_e4m3_in_place(unsigned char* stage, int row0, int row1,
                                                    int lane) {
  constexpr int RPP = 512 / D;
  constexpr int U = (D == 128) ? 4 : 2;
  constexpr int HALF = BLOCK_M * 128;  // bytes of one d half of a tile
  constexpr int SRC8 = (D / 64) * HALF - BLOCK_N * D;
  int r0, c;
  if constexpr (D == 128) {
    r0 = ((lane >> 4) << 1) | ((lane >> 2) & 1);
    c = ((((lane >> 2) ^ (lane >> 3)) & 1) << 2) | (lane & 3);
  } else {
    r0 = lane >> 2;
    c = lane & 3;
  }
  const int ps0 = row0 / RPP, ps1 = row1 / RPP;
  const unsigned char* src0 = stage + SRC8 + r0 * D + c * 16;
  unsigned char* dst0 = stage + (c >> 2) * HALF + r0 * 128;
  const int cc = 2 * (c & 3);
  for (int ps = ps0; ps < ps1; ps += U) {
    uint4 w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) w[u] = *reinterpret_cast<const uint4*>(src0 + (ps + u) * RPP * D);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const unsigned v[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
      unsigned h[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[2 * e] = e4m3x2_to_f16x2(v[e]);
        h[2 * e + 1] = e4m3x2_to_f16x2(v[e] >> 16);
      }
      // ps * RPP is a multiple of 8: the row's swizzle phase is that of
      // r0 + u * RPP
      const int sw = (r0 + u * RPP) & 7;
      unsigned char* rowp = dst0 + (ps + u) * RPP * 128;
      *reinterpret_cast<uint4*>(rowp + ((cc ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(rowp + (((cc + 1) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
    __syncwarp();
  }
}

// Converts a Q tile (bf16, as TMA loaded it: DH 128-byte-swizzled d halves)
// to f16 in place for the f16 MMAs of an e4m3 call at d 64, once its copy has
// landed (q_full at `parity`): an elementwise change, so the layout stays.
// Thread t of the softmax warpgroup takes row t (the row whose scores it
// owns) and scales it by the power of two sc that puts its largest magnitude
// in [2^7, 2^8), so no bf16 value leaves f16's range (exact down to 2^-21 of
// the row maximum); `inv` returns 1 / sc, by which the row's scores are
// scaled back.  Each warp then arrives on q_conv.
template <int DH>
__device__ __forceinline__ bool convert_q_tile(unsigned char* q, uint64_t* q_full,
                                               uint64_t* q_conv, unsigned parity, int t,
                                               unsigned* status, volatile int* abort_flag,
                                               float& inv) {
  if (!__all_sync(0xffffffffu, mbar_wait(q_full, parity, status, abort_flag))) return false;
  constexpr int HALF = BLOCK_M * 128;
  unsigned char* row = q + t * 128;
  const int sw = t & 7;
  // two passes over the row's 16-byte pieces (the maximum, then the
  // conversion, each piece written where it was read)
  unsigned m = 0;
#pragma unroll
  for (int i = 0; i < 8 * DH; ++i) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + (i >> 3) * HALF + (((i & 7) ^ sw) << 4));
    const unsigned v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) m = max(m, max(v[e] & 0x7fffu, (v[e] >> 16) & 0x7fffu));
  }
  float sc;
  split_scale(static_cast<int>(m >> 7), sc, inv);
#pragma unroll
  for (int i = 0; i < 8 * DH; ++i) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + (i >> 3) * HALF + (((i & 7) ^ sw) << 4));
    const unsigned v[4] = {w.x, w.y, w.z, w.w};
    unsigned h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      h[e] = pack2<true>(__uint_as_float(v[e] << 16) * sc, __uint_as_float(v[e] & 0xffff0000u) * sc);
    *reinterpret_cast<uint4*>(row + (i >> 3) * HALF + (((i & 7) ^ sw) << 4)) =
        make_uint4(h[0], h[1], h[2], h[3]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if ((t & 31) == 0) mbar_arrive(q_conv);
  return true;
}

// An e4m3 call at d 128 computes the scores with 8-bit MMAs straight from the
// cache's K codes.  Q (bf16, as TMA loaded it: two 128-byte-swizzled d halves)
// is split in place, once its copy has landed (q_full at `parity`), into two
// e4m3 tiles, hi over d half 0's bytes and lo over d half 1's, each 128 rows of
// 128 codes in the 128-byte-swizzled K-major layout.  Thread t of the softmax
// warpgroup takes row t (the row whose scores it owns): it reads the whole row
// before writing it, so no other thread's bytes are touched.  The row is
// scaled by the power of two sc that puts its largest magnitude in [128, 256)
// (exact), so q = (hi + lo) / sc wherever a value sits within 2^9 of the row
// maximum (below that its error is under 2^-16 of the maximum); `inv` returns
// 1 / sc, by which the row's scores are scaled back.  Each warp then arrives
// on q_conv.
__device__ __forceinline__ bool split_q_tile(unsigned char* q, uint64_t* q_full, uint64_t* q_conv,
                                             unsigned parity, int t, unsigned* status,
                                             volatile int* abort_flag, float& inv) {
  if (!__all_sync(0xffffffffu, mbar_wait(q_full, parity, status, abort_flag))) return false;
  constexpr int HALF = BLOCK_M * 128;
  unsigned char* row = q + t * 128;
  const int sw = t & 7;
  uint4 w[16];  // chunk c of d half h (elements 64h + 8c ... + 7) at w[8h + c]
#pragma unroll
  for (int i = 0; i < 16; ++i)
    w[i] = *reinterpret_cast<const uint4*>(row + (i >> 3) * HALF + (((i & 7) ^ sw) << 4));
  // bf16 magnitudes compare as unsigned integers once the sign bit is cleared
  unsigned m_lo = 0, m_hi = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const unsigned v[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      m_lo = max(m_lo, v[e] & 0x7fffu);
      m_hi = max(m_hi, v[e] & 0x7fff0000u);
    }
  }
  const int eb = static_cast<int>(max(m_lo, m_hi >> 16) >> 7);  // exponent field of the max
  float sc;
  split_scale(eb, sc, inv);  // max * sc in [2^7, 2^8)
  // A row holding an inf or a NaN (exponent field 255) gets NaN codes, so its
  // scores and output are NaN as the definition gives (the saturating
  // conversion would turn an inf into a finite code).
  const unsigned nan_row = (eb == 255) ? 0x7f7f7f7fu : 0u;
  // code chunk c (elements 16c ... 16c + 15) comes from bf16 chunks 2(c % 4)
  // and 2(c % 4) + 1 of d half c / 4
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 a = w[8 * (c >> 2) + 2 * (c & 3)], b = w[8 * (c >> 2) + 2 * (c & 3) + 1];
    const unsigned v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    unsigned hi[8], lo[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) split_pair(v[e], sc, hi[e], lo[e]);
    const int pos = (c ^ sw) << 4;
    *reinterpret_cast<uint4*>(row + pos) =
        make_uint4(hi[0] | (hi[1] << 16) | nan_row, hi[2] | (hi[3] << 16) | nan_row,
                   hi[4] | (hi[5] << 16) | nan_row, hi[6] | (hi[7] << 16) | nan_row);
    *reinterpret_cast<uint4*>(row + HALF + pos) =
        make_uint4(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16), lo[4] | (lo[5] << 16),
                   lo[6] | (lo[7] << 16));
  }
  fence_proxy_async_smem();
  __syncwarp();
  if ((t & 31) == 0) mbar_arrive(q_conv);
  return true;
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

// The weights 2^(x sl2 - ref) of 32 scores, packed in pairs (bf16, or f16
// when F16) as P; returns their sum.
template <bool F16>
__device__ __forceinline__ float exp_piece(const float (&x)[32], float sl2, float ref,
                                           unsigned (&pk)[16]) {
  const float neg_m = -ref;
  float ps0 = 0.f, ps1 = 0.f, ps2 = 0.f, ps3 = 0.f;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    float a0 = x[e], a1 = x[e + 1], a2 = x[e + 2], a3 = x[e + 3];
    ffma2(a0, a1, sl2, neg_m);
    ffma2(a2, a3, sl2, neg_m);
    a0 = fast_exp2(a0);
    a1 = fast_exp2(a1);
    a2 = fast_exp2(a2);
    a3 = fast_exp2(a3);
    fadd2(ps0, ps1, a0, a1);
    fadd2(ps2, ps3, a2, a3);
    pk[e / 2] = pack2<F16>(a0, a1);
    pk[e / 2 + 1] = pack2<F16>(a2, a3);
  }
  return (ps0 + ps1) + (ps2 + ps3);
}

// One work item: a 128-row query tile (two sub-tiles) of one request, one head
// pair (or head) and one key chunk, read from the LPT-ordered tile list.
struct Item {
  int r, qt, t0, q_len, s, chunk, pidx;
  bool live;
};

__device__ __forceinline__ Item load_item(const Problem& p, int item, int n_items, int NP,
                                          int KC) {
  Item it;
  it.live = item < n_items;
  it.r = it.qt = it.t0 = it.q_len = it.s = it.chunk = it.pidx = 0;
  if (it.live) {
    it.chunk = item % KC;
    it.pidx = (item / KC) % NP;
    const int2 tl = p.tiles[(item / KC) / NP];
    it.r = tl.x;
    it.qt = tl.y;
    it.t0 = p.qsl[it.r];
    it.q_len = p.qsl[it.r + 1] - it.t0;
    it.s = p.seq_lens[it.r];
  }
  return it;
}

// Sub-tile X of an item and the key tiles [x0, x1) it visits.
__device__ __forceinline__ Sub make_sub(const Problem& p, const Item& it, bool head_pairs, int X) {
  const int ctx = it.s - it.q_len;
  const int W = p.window;
  Sub u;
  u.h = head_pairs ? 2 * it.pidx + X : it.pidx;
  u.i0 = head_pairs ? it.qt * BLOCK_M : it.qt * 2 * BLOCK_M + X * BLOCK_M;
  u.valid = it.live && u.i0 < it.q_len;
  u.i_last = min(it.q_len, u.i0 + BLOCK_M) - 1;
  const int lo = (W > 0) ? max(0, ctx + u.i0 - W + 1) : 0;
  const int hi = p.causal ? min(it.s, ctx + u.i_last + 1) : it.s;
  u.x0 = lo / BLOCK_N;
  u.x1 = u.valid ? max(u.x0, (hi + BLOCK_N - 1) / BLOCK_N) : u.x0;
  if (p.kv_chunks > 1) {  // this item's chunk of the request's key tiles
    const int per = ((it.s + BLOCK_N - 1) / BLOCK_N + p.kv_chunks - 1) / p.kv_chunks;
    u.x0 = max(u.x0, it.chunk * per);
    u.x1 = max(u.x0, min(u.x1, (it.chunk + 1) * per));
  }
  if (!u.valid) u.x0 = u.x1 = 0;
  return u;
}

// Key tiles [u0, u0 + n) that either sub-tile visits (the two ranges touch or
// overlap); a sub-tile without key tiles does not widen the range.
__device__ __forceinline__ int union_tiles(const Sub& a, const Sub& b, int& u0) {
  const bool ha = a.x1 > a.x0, hb = b.x1 > b.x0;
  u0 = ha ? (hb ? min(a.x0, b.x0) : a.x0) : b.x0;
  const int u1 = ha ? (hb ? max(a.x1, b.x1) : a.x1) : b.x1;
  return u1 - u0;
}

// HALF: q, the cache and out are f16 (else bf16).  FP8: an e4m3 cache with
// bf16 q and out.  V tiles are widened to f16 in shared memory (exact: every
// e4m3 value is an f16 value) and P V runs in f16.  At d 128 the score MMAs
// take the K codes as they are against each Q tile split in place into e4m3
// hi and lo codes; at d 64 K tiles are widened too and each Q tile is scaled
// and converted to f16 in place.  The per-row scale of Q, the K scale and
// sl2 make the row's score scale; the V scale is out_scale.
//
// Persistent: the grid holds at most one CTA per SM; its items come from the
// LPT-ordered list, in a fixed order for the first rounds and claimed as
// CTAs get free for the last ones (warp 8 posts them in the item ring, see
// claim below).  Every role
// walks the same item sequence and keeps its ring stages and barrier phases as
// running counts across items, so the next item's Q, K and first scores go out
// while the last P V and the epilogue of the current one run.  Two orderings
// carry across an item boundary: Q is reloaded only after the q_empty commit
// that follows the item's last S MMA, and the first P V of the next item
// (which overwrites O) waits on p_full, which the softmax warps arrive on only
// after their epilogue has read O.
template <int D, bool HALF, bool FP8, bool TWO>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_kernel(const __grid_constant__ Problem p, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, float sl2, float out_scale) {
  // e4m3 at d 128: the score MMAs read the cache's K codes as they are (8-bit
  // MMAs against the split Q), so only V tiles are widened
  constexpr bool NK = FP8 && D == 128;
  using C = PrefillCfg<D, NK>;
  constexpr bool MMA_F16 = HALF || FP8;  // operand and P type of the P V MMAs
  constexpr int VST = C::VST;
  constexpr int V_SPLIT = 80;  // NK: first V row that warp 8 widens
  static_assert(!(FP8 && D != 128 && TWO), "an e4m3 call at d 64 has one MMA issuer");
  static_assert(!NK || TWO, "the 8-bit score MMAs are issued by the two-issuer loop");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::BAR_OFF);
  unsigned* status = &p.hdr->status;

  const bool head_pairs = (p.G % 2) == 0;
  const int NP = head_pairs ? p.H / 2 : p.H;
  const int KC = p.kv_chunks;
  const int n_items = p.hdr->num_prefill_tiles * NP * KC;
  // In a co-scheduled mixed batch the plan kernel keeps only prefill_ctas of
  // the grid's CTAs (one per SM); the others leave at once, and the decode
  // kernel runs on their SMs.
  const int keep = p.hdr->prefill_ctas;
  const int GS = (keep > 0 && keep < static_cast<int>(gridDim.x)) ? keep : static_cast<int>(gridDim.x);
  // The decode kernel of the same call reads nothing this kernel writes.
  if (p.pdl_trigger && threadIdx.x == 0) grid_dep_trigger();
  if (static_cast<int>(blockIdx.x) >= n_items || static_cast<int>(blockIdx.x) >= GS) return;

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
      mbar_init(&bars->k_empty[i], TWO ? 2 : 1);
    }
    // an e4m3 V tile at d 128 is announced by both producers (each widens
    // part of it)
    for (int i = 0; i < VST; ++i) {
      mbar_init(&bars->v_full[i], NK ? 2 : 1);
      mbar_init(&bars->v_empty[i], TWO ? 2 : 1);
    }
    mbar_init(&bars->q_empty, TWO ? 2 : 1);
    mbar_init(&bars->tok[0], 1);
    mbar_init(&bars->tok[1], 1);
    for (int i = 0; i < PF_KST; ++i) mbar_init(&bars->k_land[i], 1);
    for (int i = 0; i < VST; ++i) mbar_init(&bars->v_land[i], 1);
    mbar_init(&bars->q_conv[0], 4);  // one arrival per warp of the softmax warpgroup
    mbar_init(&bars->q_conv[1], 4);
    mbar_init(&bars->drain, TWO ? 2 : 1);
    // the item ring: posted by warp 8; taken by warp 10, each MMA issuer and
    // each softmax warp
    for (int i = 0; i < PF_RING; ++i) {
      mbar_init(&bars->ring_full[i], 1);
      mbar_init(&bars->ring_empty[i], 1 + (TWO ? 2 : 1) + 8);
    }
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

  // The CTA's k-th item, from the longest-first list.  The first rounds
  // follow a fixed order: CTA b takes items b, 2G-1-b, 2G+b, ... (G = GS; the
  // order snakes so that no CTA draws the heaviest item of every round).  The
  // last DYN_ROUNDS rounds' worth of items go to whichever CTA asks first:
  // warp 8 claims each with an atomic on the workspace counter (the plan
  // kernel zeroes it), so CTAs that ran ahead take more of the tail.  Warp 8
  // claims one item ahead and posts the index in the item ring, where the
  // other roles take it.  An index of n_items or more ends the CTA's
  // sequence.  A wait that gives up returns -1.
  const int rounds = (n_items + GS - 1) / GS;
  const int fixed_rounds = max(0, rounds - DYN_ROUNDS);
  auto claim = [&](int k) -> int {  // warp 8, one thread
    int idx = (k < fixed_rounds)
                  ? k * GS + ((k & 1) ? GS - 1 - static_cast<int>(blockIdx.x)
                                      : static_cast<int>(blockIdx.x))
                  : fixed_rounds * GS + static_cast<int>(atomicAdd(&p.hdr->next_item, 1u));
    idx = min(idx, n_items);
    const int slot = k % PF_RING;
    if (k >= PF_RING &&
        !mbar_wait(&bars->ring_empty[slot], ((k / PF_RING) - 1) & 1, status, abort_flag))
      return -1;
    bars->ring[slot] = idx;
    mbar_arrive(&bars->ring_full[slot]);
    return idx;
  };
  auto take = [&](int k) -> int {  // every other role: one thread, or all lanes of a warp
    const int slot = k % PF_RING;
    if (!mbar_wait(&bars->ring_full[slot], (k / PF_RING) & 1, status, abort_flag)) return -1;
    return *reinterpret_cast<volatile int*>(&bars->ring[slot]);
  };
  auto release = [&](int k) { mbar_arrive(&bars->ring_empty[k % PF_RING]); };

  unsigned char* sQ = smem + C::Q_OFF;
  unsigned char* sK = smem + C::K_OFF;
  unsigned char* sV = smem + C::V_OFF;
  const int rows_box = p.bs < BLOCK_N ? p.bs : BLOCK_N;  // rows of one cache copy
  const int pages_per_tile = BLOCK_N / rows_box;         // copies of one key tile

  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(other_regs(FP8)));
  if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ TMA producers
    // Warp 8 streams the Q tiles and the K tiles, warp 10 the V tiles, each
    // through its own ring, so a K tile never queues behind a V slot.  Each
    // warp reads the block ids of a key tile in one coalesced load, one tile
    // ahead.  Lane 0 waits for the stage and posts the tile's bytes; the
    // tile's copies (one per page and d half) then go out from one lane each,
    // so a tile costs one copy instruction, not 2 x pages of them in one
    // thread.
    const int kv = (warp == 10) ? 1 : 0;
    const int nst = kv ? VST : PF_KST;
    unsigned char* ring = kv ? sV : sK;
    const int stage_bytes = kv ? C::TILE : C::KSTAGE;
    // Copy `lane` of a tile: a K copy is page lane / DH, d half lane % DH (an
    // e4m3 K tile at d 128 is one 128-byte column block: DHK = 1); a 16-bit V
    // copy is the whole of page lane (its rows_box / 16 groups).
    constexpr int DHK = NK ? 1 : C::DH;
    const bool v16 = kv && !FP8;
    const int my_pg = v16 ? lane : lane / DHK, my_dh = v16 ? 0 : lane % DHK;
    // the tiles this warp copies as they are (else as e4m3 rows to be widened)
    const bool direct = !FP8 || (NK && kv == 0);
    if (kv == 0 && lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    int jg = 0;        // key tiles streamed so far (ring position)
    int n_worked = 0;  // items with at least one key tile so far
    // For the drain after a wait gave up: ring positions [0, armed_end) had
    // their bytes posted; Q tiles of sub-tile X were posted q_arms_X times.
    int armed_end = 0, q_arms0 = 0, q_arms1 = 0;
    bool gave_up = false;
#ifdef PATTN_WAIT_TEST
    const int skip_pos = (!FP8 && p.test_skip == 1 && kv == 0 && blockIdx.x == 0) ? 0 : -1;
#else
    constexpr int skip_pos = -1;
#endif
    // Warp 8 claims the next item as it starts the current one (its metadata
    // then loads in the shadow of this item); warp 10 takes the items from the
    // ring, one ahead as well.
    auto next_index = [&](int k) {
      int idx = 0;
      if (lane == 0) {
        if (kv == 0) {
          idx = claim(k);
        } else {
          idx = take(k);
          if (idx >= 0) release(k);
        }
      }
      return __shfl_sync(FULL, idx, 0);
    };
    int idx_next = next_index(0);
    if (idx_next < 0) gave_up = true;
    Item nxt = load_item(p, gave_up ? n_items : idx_next, n_items, NP, KC);
    for (int k = 0; !gave_up && nxt.live; ++k) {
      const Item it = nxt;
      idx_next = next_index(k + 1);
      if (idx_next < 0) {
        gave_up = true;
        break;
      }
      nxt = load_item(p, idx_next, n_items, NP, KC);
      const Sub subA = make_sub(p, it, head_pairs, 0), subB = make_sub(p, it, head_pairs, 1);
      int u0;
      const int n_union = union_tiles(subA, subB, u0);
      if (n_union <= 0) continue;
      const int g = subA.h / p.G;
      const int s = it.s;
      int ok = 1;
      if (kv == 0 && lane == 0) {
        // Q buffers are free once every S MMA of the previous item is done.
        if (n_worked > 0 && !mbar_wait(&bars->q_empty, (n_worked - 1) & 1, status, abort_flag))
          ok = 0;
#pragma unroll
        for (int X = 0; X < 2; ++X) {
          const Sub& u = X ? subB : subA;
          if (!ok || u.x1 <= u.x0) continue;
          mbar_arrive_expect_tx(&bars->q_full[X], C::TILE);
          ++(X ? q_arms1 : q_arms0);
#pragma unroll
          for (int dh = 0; dh < C::DH; ++dh)
            tma_load_3d(sQ + X * C::TILE + dh * C::HALF, &qmap, &bars->q_full[X], dh * 64, u.h,
                        it.t0 + u.i0);
        }
      }
      ok = __shfl_sync(FULL, ok, 0);
      if (!ok) {
        gave_up = true;
        break;
      }
      const int* bt = p.block_table + static_cast<int64_t>(it.r) * p.bt_stride;
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
      if (NK && kv == 0) {
        // e4m3 at d 128: the K codes go straight to their stage (one
        // 128-byte-swizzled column block), PF_KST - 1 tiles ahead, and
        // between copies this warp widens rows [V_SPLIT, BLOCK_N) of each V
        // tile (warp 10 rows [0, V_SPLIT)).  The copy of tile j + PF_KST - 1
        // waits for the scores of tile j - 1, whose MMAs need only V tiles
        // before j - 1, so the two jobs never wait on each other.
        int blk_next = page_block(u0);
        int n_issued = 0;
        auto issue_k = [&]() {
          const int kt = u0 + n_issued, jt = jg + n_issued;
          const int key_base = kt * BLOCK_N;
          const int my_blk = __shfl_sync(FULL, blk_next, lane);
          if (n_issued + 1 < n_union) blk_next = page_block(kt + 1);
          const int n_load = min(pages_per_tile, (s - key_base + rows_box - 1) / rows_box);
          const int my_key0 = key_base + lane * rows_box;
          const int my_slot = p.bs_shift >= 0 ? (my_key0 & (p.bs - 1)) : (my_key0 % p.bs);
          const int st = jt % PF_KST;
          int good = 1;
          if (lane == 0) {
            if (jt >= PF_KST && !mbar_wait(&bars->k_empty[st], ((jt / PF_KST) - 1) & 1, status,
                                           abort_flag))
              good = 0;
            else
              mbar_arrive_expect_tx(&bars->k_full[st],
                                    static_cast<unsigned>(n_load * rows_box * 128));
          }
          good = __shfl_sync(FULL, good, 0);
          if (!good) return 0;
          armed_end = jt + 1;
          if (lane < n_load)
            tma_load_4d(sK + st * C::KSTAGE + lane * rows_box * 128, &kmap, &bars->k_full[st], 0,
                        g, my_slot, my_blk);
          ++n_issued;
          return 1;
        };
        while (ok && n_issued < min(PF_KST - 1, n_union)) ok = issue_k();
        for (int j = 0; ok && j < n_union; ++j) {
          if (n_issued < n_union && !(ok = issue_k())) break;
          const int jt = jg + j, st = jt % VST;
          if (!__all_sync(FULL, mbar_wait(&bars->v_land[st], (jt / VST) & 1, status, abort_flag))) {
            ok = 0;
            break;
          }
          const int key_base = (u0 + j) * BLOCK_N;
          const int rows = min(pages_per_tile, (s - key_base + rows_box - 1) / rows_box) * rows_box;
          widen_e4m3_in_place<D>(sV + st * C::TILE, V_SPLIT, max(rows, V_SPLIT), lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->v_full[st]);
        }
        jg += n_union;
      } else if (direct) {
        int blk_next = page_block(u0);
        for (int j = 0; j < n_union; ++j, ++jg) {
          const int key_base = (u0 + j) * BLOCK_N;
          const int my_blk = __shfl_sync(FULL, blk_next, my_pg);
          if (j + 1 < n_union) blk_next = page_block(u0 + j + 1);
          // pages of this tile that hold keys below seq_len
          const int n_load = min(pages_per_tile, (s - key_base + rows_box - 1) / rows_box);
          const int my_key0 = key_base + my_pg * rows_box;
          const int my_slot = p.bs_shift >= 0 ? (my_key0 & (p.bs - 1)) : (my_key0 % p.bs);
          const int st = jg % nst;
          uint64_t* empty = kv ? &bars->v_empty[st] : &bars->k_empty[st];
          uint64_t* full = kv ? &bars->v_full[st] : &bars->k_full[st];
          const unsigned bytes = static_cast<unsigned>(n_load * rows_box * 128 * DHK);
          // (wait-test build: the skipped position posts no bytes and issues
          // no copy, so the MMA thread's wait for it runs out)
          const bool skip = jg == skip_pos;
          if (lane == 0) {
            if (jg >= nst && !mbar_wait(empty, ((jg / nst) - 1) & 1, status, abort_flag))
              ok = 0;
            else if (!skip)
              mbar_arrive_expect_tx(full, bytes);
          }
          ok = __shfl_sync(FULL, ok, 0);
          if (!ok) break;
          armed_end = jg + 1;
          if (my_pg < n_load && !skip) {
            if (v16)
              tma_load_5d(ring + st * stage_bytes + my_pg * (C::DH * rows_box * 128), &vmap, full, 0,
                          0, 0, g, (p.NB + my_blk) * (p.bs >> 4) + (my_slot >> 4));
            else
              tma_load_4d(ring + st * stage_bytes + my_dh * C::HALF + my_pg * rows_box * 128, &kmap,
                          full, my_dh * 64, g, my_slot, my_blk);
          }
        }
      } else {
        // e4m3 (V tiles, and K tiles at d 64): a tile's pages land as bytes
        // at the top of its ring stage (the last BLOCK_N x D bytes, rows of D
        // bytes, no swizzle; the map in vmap), where the warp
        // widens them in place into the swizzled f16 tile TMA would have
        // written, then announces the stage with a plain arrival.  Copies run
        // nst - 1 tiles ahead of the widening: after widening tile j the warp
        // waits for the stage of tile j - 1 and refills it with tile
        // j + nst - 1.  They stop at the item's last tile.
        uint64_t* lands = kv ? bars->v_land : bars->k_land;
        auto issue = [&](int jt, int kt, int blkv) {
          const int key_base = kt * BLOCK_N;
          const int n_load = min(pages_per_tile, (s - key_base + rows_box - 1) / rows_box);
          const int st = jt % nst;
          uint64_t* empty = kv ? &bars->v_empty[st] : &bars->k_empty[st];
          int good = 1;
          if (lane == 0) {
            if (jt >= nst && !mbar_wait(empty, ((jt / nst) - 1) & 1, status, abort_flag))
              good = 0;
            else
              mbar_arrive_expect_tx(&lands[st], static_cast<unsigned>(n_load * rows_box * D));
          }
          good = __shfl_sync(FULL, good, 0);
          if (good) armed_end = jt + 1;
          if (good && lane < n_load) {
            const int key0 = key_base + lane * rows_box;
            const int slot = p.bs_shift >= 0 ? (key0 & (p.bs - 1)) : (key0 % p.bs);
            tma_load_4d(ring + st * stage_bytes + C::SRC8 + lane * rows_box * D, &vmap, &lands[st],
                        0, g, slot, kv * p.NB + blkv);
          }
          return good;
        };
        int blk_next = page_block(u0);
        int n_issued = 0;
        auto issue_next = [&]() {
          const int blk = blk_next;
          if (n_issued + 1 < n_union) blk_next = page_block(u0 + n_issued + 1);
          const int good = issue(jg + n_issued, u0 + n_issued, blk);
          ++n_issued;
          return good;
        };
        while (ok && n_issued < min(nst - 1, n_union)) ok = issue_next();
        for (int j = 0; ok && j < n_union; ++j) {
          const int jt = jg + j, st = jt % nst;
          if (!__all_sync(FULL, mbar_wait(&lands[st], (jt / nst) & 1, status, abort_flag))) {
            ok = 0;
            break;
          }
          const int key_base = (u0 + j) * BLOCK_N;
          const int n_load = min(pages_per_tile, (s - key_base + rows_box - 1) / rows_box);
          widen_e4m3_in_place<D>(ring + st * stage_bytes, 0,
                                 NK ? min(n_load * rows_box, V_SPLIT) : n_load * rows_box, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(kv ? &bars->v_full[st] : &bars->k_full[st]);
          if (n_issued < n_union) ok = issue_next();
        }
        jg += n_union;
      }
      if (!ok) {
        gave_up = true;
        break;
      }
      ++n_worked;
    }
    // A role gave up on a wait: no copy this warp armed may still be writing
    // shared memory when the CTA frees its resources and exits.
    if (gave_up || *abort_flag) {
      if (lane == 0) {
        uint64_t* armed = !direct ? (kv ? bars->v_land : bars->k_land)
                                  : (kv ? bars->v_full : bars->k_full);
        drain_armed(armed, nst, armed_end, skip_pos, status);
        if (kv == 0) {
          if (q_arms0 > 0) mbar_wait(&bars->q_full[0], (q_arms0 - 1) & 1, status, nullptr);
          if (q_arms1 > 0) mbar_wait(&bars->q_full[1], (q_arms1 - 1) & 1, status, nullptr);
        }
      }
      __syncwarp();
    }
  } else if (warp == 9 || (TWO && warp == 11)) {
    // ------------------------------------------------------------ MMA issuers
    // A tcgen05.mma occupies its issuing thread for about as long as the
    // tensor core takes to run it, so everything else that thread does (barrier
    // waits, commits, bookkeeping) leaves the tensor core idle.  With TWO
    // (a 16-bit cache, or e4m3 at d 128) two threads issue: warp 9 sub-tile
    // A's MMAs, warp 11 sub-tile B's.  They take turns, A then B for each key
    // tile, handing a token over through tok[] (A's turn t waits for B's turn
    // t - 1, B's turn t for A's turn t), and each waits for its operands and
    // commits while the other one issues.  Each commits its own release of
    // every K and V stage and of the Q tiles (those barriers then count one
    // arrival per issuer).  Otherwise (an e4m3 cache at d 64) warp 9 issues
    // both sub-tiles' MMAs in the same order.
    if (lane == 0) {
      constexpr unsigned idesc_s = make_idesc_f16(BLOCK_M, BLOCK_N, !MMA_F16, false);
      // e4m3 x e4m3 (type fields 0), fp32 accumulation, both K-major
      constexpr unsigned idesc_s8 = make_idesc_f16(BLOCK_M, BLOCK_N, false, false);
      constexpr unsigned idesc_pv = make_idesc_f16(BLOCK_M, D, !MMA_F16, true);
      // Base descriptors; a byte offset o moves the start address field by
      // o >> 4 (shared addresses stay far below the field's 256 KB range).
      const uint64_t q_d = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t k_d = smem_desc_sw128(smem_u32(sK), 16, 1024);
      // V: the d halves of a group of V_ROWS keys are V_ROWS x 128 bytes apart
      constexpr int V_ROWS = v_rows<FP8>();
      const uint64_t v_d = smem_desc_sw128(smem_u32(sV), V_ROWS * 128, 1024);
      if constexpr (TWO) {
        // This thread issues sub-tile X's MMAs.
        const int X = (warp == 11) ? 1 : 0;
        int jg = 0;         // key tiles consumed so far (ring position)
        int pv_tot = 0;     // P V of sub-tile X so far (p_full phase)
        int q_tot = 0;      // Q tiles of sub-tile X so far (q_full phase)
        unsigned turn = 0;  // turns taken so far
        bool ok = true;
        for (int k = 0; ok; ++k) {
          const int idx = take(k);
          if (idx < 0) {
            ok = false;
            break;
          }
          release(k);
          const Item it = load_item(p, idx, n_items, NP, KC);
          if (!it.live) break;
          const Sub subA = make_sub(p, it, head_pairs, 0), subB = make_sub(p, it, head_pairs, 1);
          int u0;
          const int n_union = union_tiles(subA, subB, u0);
          if (n_union <= 0) continue;
          const Sub u = X ? subB : subA;
          int n_pv = 0;
          bool q_ready = false;
          for (int j = 0; ok && j <= n_union; ++j, ++turn) {
            const int kt = u0 + j;
            const int jj = jg + j;
            const bool do_pv = j >= 1 && u.active(kt - 1);  // P V for the previous key tile
            const bool do_s = j < n_union && u.active(kt);  // scores for this key tile
            const int stp = (jj - 1) % VST;
            const int st = jj % PF_KST;
            // The operands, all before the turn: P and V of the previous
            // tile, K of this tile and Q.
            if (do_pv && !(mbar_wait(&bars->p_full[X], pv_tot & 1, status, abort_flag) &&
                           mbar_wait(&bars->v_full[stp], ((jj - 1) / VST) & 1, status,
                                     abort_flag))) {
              ok = false;
              break;
            }
            if (do_s) {
              if (!mbar_wait(&bars->k_full[st], (jj / PF_KST) & 1, status, abort_flag)) {
                ok = false;
                break;
              }
              if (!q_ready) {
                // an e4m3 call's Q is usable once its softmax warpgroup has split it
                if (!mbar_wait(FP8 ? &bars->q_conv[X] : &bars->q_full[X], q_tot & 1, status,
                               abort_flag)) {
                  ok = false;
                  break;
                }
                q_ready = true;
                ++q_tot;
              }
            }
            // The turn: A's turn t follows B's turn t - 1, B's turn t follows
            // A's turn t.
            if ((X == 1 || turn > 0) &&
                !mbar_wait(&bars->tok[X], (X ? turn : turn - 1) & 1, status, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // Both blocks' base addresses are ready before the first MMA, so
            // nothing but MMAs runs between them; they are made opaque so that
            // their per-MMA offsets are added at each use instead of being
            // hoisted out of the loops as live registers.
            uint64_t qb = q_d + ((X * C::TILE) >> 4);
            unsigned s_t = tmem + C::s_col(X);
            const uint64_t kb = k_d + ((st * C::KSTAGE) >> 4);
            unsigned p_t = tmem + C::s_col(X);
            unsigned o_t = tmem + C::o_col(X);
            const uint64_t vb = v_d + ((stp * C::TILE) >> 4);
            asm volatile("" : "+l"(qb), "+r"(s_t), "+r"(p_t), "+r"(o_t));
            if (do_pv) {
#pragma unroll
              for (int kk = 0; kk < BLOCK_N / 16; ++kk)
                tc_mma_ts(o_t, p_t + kk * 8,
                          vb + ((((kk * 16) / V_ROWS * C::DH * V_ROWS) + (kk * 16) % V_ROWS) *
                                    128 >> 4),
                          idesc_pv, (n_pv > 0 || kk > 0) ? 1u : 0u);
            }
            if (do_s) {
              if constexpr (NK) {
                // Q hi (d half 0's bytes) then Q lo (d half 1's), each against
                // the K codes in four 32-code steps
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  tc_mma_ss_f8(s_t, qb + (((kk >> 2) * C::HALF + (kk & 3) * 32) >> 4),
                               kb + (((kk & 3) * 32) >> 4), idesc_s8, kk > 0 ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const unsigned off = ((kk >> 2) * C::HALF + (kk & 3) * 32) >> 4;
                  tc_mma_ss(s_t, qb + off, kb + off, idesc_s, kk > 0 ? 1u : 0u);
                }
              }
            }
            mbar_arrive(&bars->tok[1 - X]);  // the other issuer's turn
            if (do_pv) {
              ++n_pv;
              ++pv_tot;
            }
            // Commits, while the other issuer's MMAs run.  Every stage of the
            // item's key tiles is released by both issuers.
            if (do_s) tc_commit(&bars->s_full[X]);
            if (do_pv && kt - 1 == u.x1 - 1) tc_commit(&bars->o_final[X]);
            if (j >= 1) tc_commit(&bars->v_empty[stp]);
            if (j < n_union) tc_commit(&bars->k_empty[st]);
            // every S of this item is issued: its Q tiles may be replaced
            if (j == n_union - 1) tc_commit(&bars->q_empty);
          }
          jg += n_union;
        }
        // No MMA may still be running when TMEM is released (matters only when
        // a role gave up on a wait); both issuers arrive on drain.
        tc_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, status, nullptr);
      } else {
        int jg = 0;                  // key tiles consumed so far (ring position)
        int pv_tot0 = 0, pv_tot1 = 0;  // P V of sub-tile X so far (p_full phase)
        int q_tot0 = 0, q_tot1 = 0;    // Q tiles of sub-tile X so far (q_full phase)
        bool issued = false, ok = true;
        for (int k = 0; ok; ++k) {
          const int idx = take(k);
          if (idx < 0) {
            ok = false;
            break;
          }
          release(k);
          const Item it = load_item(p, idx, n_items, NP, KC);
          if (!it.live) break;
          const Sub subA = make_sub(p, it, head_pairs, 0), subB = make_sub(p, it, head_pairs, 1);
          int u0;
          const int n_union = union_tiles(subA, subB, u0);
          if (n_union <= 0) continue;
          issued = true;
          int n_pv0 = 0, n_pv1 = 0;
          bool q_ready0 = false, q_ready1 = false;
          for (int j = 0; ok && j <= n_union; ++j) {
            const int kt = u0 + j;
            const int jj = jg + j;
            bool k_ready = false, v_ready = false;
            // Unrolled: every per-sub-tile value stays in a register (a runtime
            // choice between two locals would put them in local memory).
  #pragma unroll
            for (int X = 0; X < 2; ++X) {
              const Sub& u = X ? subB : subA;
              int& n_pv = X ? n_pv1 : n_pv0;
              int& pv_tot = X ? pv_tot1 : pv_tot0;
              int& q_tot = X ? q_tot1 : q_tot0;
              bool& q_ready = X ? q_ready1 : q_ready0;
              // P V for the previous key tile
              if (j >= 1 && u.active(kt - 1)) {
                const int stp = (jj - 1) % VST;
                if (!mbar_wait(&bars->p_full[X], pv_tot & 1, status, abort_flag)) {
                  ok = false;
                  break;
                }
                if (!v_ready) {
                  if (!mbar_wait(&bars->v_full[stp], ((jj - 1) / VST) & 1, status, abort_flag)) {
                    ok = false;
                    break;
                  }
                  v_ready = true;
                }
                tc_fence_after();
                // The base addresses are made opaque here so that their per-MMA
                // offsets are added at each use instead of being hoisted out of
                // the loops as 16 live registers.
                unsigned p_t = tmem + C::s_col(X);
                unsigned o_t = tmem + C::o_col(X);
                asm volatile("" : "+r"(p_t), "+r"(o_t));
                const uint64_t vb = v_d + ((stp * C::TILE) >> 4);
  #pragma unroll
                for (int kk = 0; kk < BLOCK_N / 16; ++kk)
                  tc_mma_ts(o_t, p_t + kk * 8,
                            vb + ((((kk * 16) / V_ROWS * C::DH * V_ROWS) + (kk * 16) % V_ROWS) *
                                      128 >> 4),
                            idesc_pv,
                            (n_pv > 0 || kk > 0) ? 1u : 0u);
                ++n_pv;
                ++pv_tot;
                if (kt - 1 == u.x1 - 1) tc_commit(&bars->o_final[X]);
                if (X == 1 || !subB.active(kt - 1)) tc_commit(&bars->v_empty[stp]);
              }
              // scores for this key tile
              if (j < n_union && u.active(kt)) {
                const int st = jj % PF_KST;
                if (!k_ready) {
                  if (!mbar_wait(&bars->k_full[st], (jj / PF_KST) & 1, status, abort_flag)) {
                    ok = false;
                    break;
                  }
                  k_ready = true;
                }
                if (!q_ready) {
                  // an e4m3 call's Q is usable once its softmax warpgroup has converted it
                  if (!mbar_wait(FP8 ? &bars->q_conv[X] : &bars->q_full[X], q_tot & 1, status,
                                 abort_flag)) {
                    ok = false;
                    break;
                  }
                  q_ready = true;
                  ++q_tot;
                }
                tc_fence_after();
                uint64_t qb = q_d + ((X * C::TILE) >> 4);
                unsigned s_t = tmem + C::s_col(X);
                asm volatile("" : "+l"(qb), "+r"(s_t));
                const uint64_t kb = k_d + ((st * C::KSTAGE) >> 4);
  #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const unsigned off = ((kk >> 2) * C::HALF + (kk & 3) * 32) >> 4;
                  tc_mma_ss(s_t, qb + off, kb + off, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(&bars->s_full[X]);
                if (X == 1 || !subB.active(kt)) tc_commit(&bars->k_empty[st]);
              }
            }
            // every S of this item is issued: its Q tiles may be replaced
            if (ok && j == n_union - 1) tc_commit(&bars->q_empty);
          }
          jg += n_union;
        }
        // No MMA may still be running when TMEM is released (matters only when
        // a role gave up on a wait).
        if (issued) {
          tc_commit(&bars->drain);
          mbar_wait(&bars->drain, 0, status, nullptr);
        }
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(softmax_regs(FP8)));
    // ------------------------------------------------------------ softmax warpgroups
    const int X = warp >> 2;            // 0: A (warps 0-3), 1: B (warps 4-7)
    const int row = threadIdx.x & 127;  // TMEM lane
    const unsigned lane_base = tmem + (static_cast<unsigned>((warp & 3) * 32) << 16);
    const unsigned s_t = lane_base + C::s_col(X);
    const unsigned o_t = lane_base + C::o_col(X);
    const int W = p.window;
    // Phases carried across items, packed in one word to spare registers:
    // bit 0 the s_full phase of this sub-tile, bit 1 its o_final phase, bits
    // 2 and up the V ring position of the key tiles so far modulo 2 x VST (a
    // V slot's stage and parity).
    constexpr unsigned VPOS = 2 * VST;
    unsigned ph = 0;
    bool ok = true;
    int qn = 0;             // Q tiles of this sub-tile converted so far (FP8)
    // Score scale of this row: sl2, over an e4m3 cache times the row's 1 / sc,
    // kept normal so that a masked score (-inf) still maps to -inf.  Set when
    // the item's Q tile is converted (the previous item no longer needs it).
    float sl2r = sl2;
    // An e4m3 call converts each item's Q tile at the end of the previous
    // item (below), so its loop starts one step early, on an empty item, to
    // convert the first one there too: one copy of that long code.
    // Each softmax warp takes every item index from the ring (all lanes wait,
    // one arrival per warp).
    auto take_warp = [&](int k) {
      const int idx = take(k);
      const bool got = __all_sync(FULL, idx >= 0);
      if (got && lane == 0) release(k);
      return got ? idx : -1;
    };
    Item it = load_item(p, n_items, n_items, NP, KC);  // none yet
    if (!FP8) {
      const int idx0 = take_warp(0);
      if (idx0 < 0) ok = false;
      else it = load_item(p, idx0, n_items, NP, KC);
    }
    for (int k = FP8 ? -1 : 0; ok && (k < 0 || it.live); ++k) {
      const Sub u = make_sub(p, it, head_pairs, X);
      const Sub subA = X ? make_sub(p, it, head_pairs, 0) : u;
      const Sub subB = X ? u : make_sub(p, it, head_pairs, 1);
      int u0;
      const int n_union = union_tiles(subA, subB, u0);
      // Per-item constants, folded so that few registers stay live through
      // the key-tile loop.  Row i of the sub-tile sees keys [kmin_row, kmax_row).
      const int s = it.s;
      const int ctx = s - it.q_len;
      const int i = u.i0 + row;
      const bool row_ok = i < it.q_len;
      const int kmax_row = p.causal ? min(s, ctx + i + 1) : s;
      const int kmin_row = (W > 0) ? ctx + i - W + 1 : -(1 << 30);
      // A tile needs the per-element mask when key0 > edge_hi (keys at or past
      // seq_len, or past the causal limit of the first row) or key0 <= edge_lo
      // (keys below the window of the last row).
      const int edge_hi = min(s - BLOCK_N, p.causal ? ctx + u.i0 - (BLOCK_N - 1) : s);
      const int edge_lo = (W > 0) ? ctx + u.i_last - W : -(1 << 30);
      // The tile holding seq_len - 1 has V rows at or past seq_len; they are
      // zeroed by the first sub-tile whose P V reads it.
      const int tail_kt = (s - 1) / BLOCK_N;
      const int vz_kt = (u.active(tail_kt) && (X == 0 || !subA.active(tail_kt))) ? tail_kt : -1;
      // its V ring position modulo 2 x VST (used only when vz_kt >= 0, where
      // tail_kt >= u0)
      const unsigned vz_m = ((ph >> 2) + static_cast<unsigned>(tail_kt - u0)) % VPOS;
      const int vz_row = s - tail_kt * BLOCK_N;                  // first row to zero
      // output row of the epilogue
      const int64_t orow_i = static_cast<int64_t>(it.t0 + i) * p.H + u.h;
      const int chunk = it.chunk;
      float m_run = -INFINITY, l_run = 0.f;
      const int nt = u.x1 - u.x0;
      for (int c = 0; c < nt; ++c) {
        const int kt = u.x0 + c;
        const int key0 = kt * BLOCK_N;
        if (!__all_sync(FULL, mbar_wait(&bars->s_full[X], (ph ^ c) & 1, status, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool edge = key0 > edge_hi || key0 <= edge_lo;
        // column limits of this row in the tile: visible iff lim_lo <= col < lim_hi
        const int lim_hi = kmax_row - key0;
        const int lim_lo = kmin_row - key0;
        // Common case: the reference stays.  The weights against it are
        // computed in registers; if any exceeded 2^RESCALE_THRESHOLD, their
        // sum did too, and the tile goes down the path below, which takes the
        // row max.  So the max is taken only for a row's first tile and for
        // the rare tile whose scores outgrow the reference.  P (16 packed
        // columns per 32 scores) is stored at columns [0, 64) only once the
        // tile is known to stay on this path, so the scores are still in TMEM
        // for the other one.
        bool slow = (m_run == -INFINITY);
        float ps = 0.f;
        if (!__any_sync(FULL, slow)) {
          float sv[BLOCK_N];
#pragma unroll
          for (int g = 0; g < BLOCK_N / 32; ++g)
            tc_ld32(s_t + g * 32, *reinterpret_cast<float(*)[32]>(&sv[g * 32]));
          tc_wait_ld();
          if (edge) {
#pragma unroll
            for (int q = 0; q < BLOCK_N; ++q)
              sv[q] = (q < lim_hi && q >= lim_lo) ? sv[q] : -INFINITY;
          }
          unsigned pk[BLOCK_N / 2];
#pragma unroll
          for (int g = 0; g < BLOCK_N / 32; ++g)
            ps += exp_piece<MMA_F16>(*reinterpret_cast<const float(*)[32]>(&sv[g * 32]), sl2r,
                                     m_run, *reinterpret_cast<unsigned(*)[16]>(&pk[g * 16]));
          slow = !(ps <= FAST_SUM_LIMIT);
          if (!__any_sync(FULL, slow)) {
#pragma unroll
            for (int g = 0; g < BLOCK_N / 32; ++g)
              tc_st16u(s_t + g * 16, *reinterpret_cast<const unsigned(*)[16]>(&pk[g * 16]));
          }
        }
        if (__any_sync(FULL, slow)) {
          // The scores again (still in TMEM: nothing was stored over them),
          // all 128 columns in one round trip.
          float sv[BLOCK_N];
#pragma unroll
          for (int g = 0; g < BLOCK_N / 32; ++g)
            tc_ld32(s_t + g * 32, *reinterpret_cast<float(*)[32]>(&sv[g * 32]));
          tc_wait_ld();
          if (edge) {
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
          const float mx_s = (mx == -INFINITY) ? -INFINITY : mx * sl2r;
          // Lazy rescale: move the reference max only when it grows by > 2^8,
          // or, for a row whose own weights summed above the limit, whenever
          // it grows (else that row would take this path on every tile).
          const bool grow = mx_s > m_run + (slow ? 0.f : RESCALE_THRESHOLD);
          const bool need_o = grow && (m_run != -INFINITY) && (c > 0);
          float alpha = 1.f;
          if (grow) {
            alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - mx_s);
            l_run *= alpha;
            m_run = mx_s;
          }
          // The weights, each 32 columns' P stored as soon as it is packed
          // (to columns [16g, 16g + 16), whose scores are in registers).
          const float ref = (m_run == -INFINITY) ? 0.f : m_run;
          ps = 0.f;
#pragma unroll
          for (int g = 0; g < BLOCK_N / 32; ++g) {
            unsigned pk[16];
            ps += exp_piece<MMA_F16>(*reinterpret_cast<const float(*)[32]>(&sv[g * 32]), sl2r,
                                     ref, pk);
            tc_st16u(s_t + g * 16, pk);
          }
          // O is rescaled last, once the score registers are free.  P V of
          // the previous tile is complete: the commit that announced these
          // scores was issued after it.
          if (__any_sync(FULL, need_o)) {
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
        }
        l_run += ps;
        tc_wait_st();

        // Zero V rows at or past seq_len before P V reads them (done by the
        // first sub-tile whose P V reads this tile).
        if (kt == vz_kt) {
          const int st = vz_m % VST;
          if (!__all_sync(FULL, mbar_wait(&bars->v_full[st], vz_m / VST, status, abort_flag))) {
            ok = false;
            break;
          }
          if (row >= vz_row) {
            // key `row` of the tile: group row / V_ROWS, row row % V_ROWS of
            // each of its d halves
            constexpr int V_ROWS = v_rows<FP8>();
            unsigned char* vrow = sV + st * C::TILE + (row / V_ROWS) * (C::DH * V_ROWS * 128) +
                                  (row % V_ROWS) * 128;
#pragma unroll
            for (int dh = 0; dh < C::DH; ++dh)
#pragma unroll
              for (int b = 0; b < 128; b += 16)
                *reinterpret_cast<uint4*>(vrow + dh * V_ROWS * 128 + b) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(&bars->p_full[X]);
      }
      ph = ((ph ^ (nt & 1)) & 3) | ((((ph >> 2) + static_cast<unsigned>(n_union)) % VPOS) << 2);
      // The next item's metadata is fetched here, where the score registers
      // are dead, and lands while the epilogue runs.
      const int idx_next = ok ? take_warp(k + 1) : -1;
      if (idx_next < 0) ok = false;
      const Item nxt = load_item(p, ok ? idx_next : n_items, n_items, NP, KC);
      if constexpr (FP8) {
        // The next item's Q tile of this sub-tile is loaded once this item's
        // last S MMA is done: split it (d 128) or convert it to f16 (d 64)
        // now, while the last P V runs, so the next item's first scores need
        // not wait for the epilogue.
        if (ok && make_sub(p, nxt, head_pairs, X).x1 > make_sub(p, nxt, head_pairs, X).x0) {
          float inv = 1.f;
          if (!(NK ? split_q_tile(sQ + X * C::TILE, &bars->q_full[X], &bars->q_conv[X], qn & 1,
                                  row, status, abort_flag, inv)
                   : convert_q_tile<C::DH>(sQ + X * C::TILE, &bars->q_full[X], &bars->q_conv[X],
                                           qn & 1, row, status, abort_flag, inv))) {
            ok = false;
          } else {
            sl2r = fmaxf(sl2 * inv, 1e-37f);
            ++qn;
          }
        }
      }

      // ---------------------------------------------------------- epilogue
      // The normalised row goes to out, or (partial-result mode) to o32 in
      // fp32 with its log2-domain lse = m + log2(l).
      const int64_t ri = orow_i * KC + chunk;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + orow_i * D;
      bool have_o = false;
      if (u.valid && ok && nt > 0) {
        have_o = __all_sync(FULL, mbar_wait(&bars->o_final[X], (ph >> 1) & 1, status, abort_flag));
        ph ^= 2;
        if (!have_o) ok = false;
      }
      if (have_o) {
        tc_fence_after();
        // a final output row includes its head's sink in the normaliser
        const float l_tot = p.o32 ? l_run : l_run + sink_term(p.sinks, u.h, m_run);
        const float inv = (l_tot > 0.f) ? out_scale / l_tot : 0.f;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          float ov[32];
          tc_ld32(o_t + q * 32, ov);
          tc_wait_ld();
          if (row_ok) {
            if (p.o32) {
              float4* dst = reinterpret_cast<float4*>(p.o32 + ri * D + q * 32);
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                dst[e / 4] =
                    make_float4(ov[e] * inv, ov[e + 1] * inv, ov[e + 2] * inv, ov[e + 3] * inv);
            } else {
              unsigned pkd[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)
                pkd[e] = pack2<HALF>(ov[2 * e] * inv, ov[2 * e + 1] * inv);
#pragma unroll
              for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<uint4*>(orow + q * 32 + e * 2) =
                    make_uint4(pkd[e], pkd[e + 1], pkd[e + 2], pkd[e + 3]);
            }
          }
        }
        if (p.o32 && row_ok) p.lse32[ri] = (l_run > 0.f) ? m_run + __log2f(l_run) : -INFINITY;
      } else if (u.valid && row_ok) {
        if (p.o32) {
          for (int e = 0; e < D; ++e) p.o32[ri * D + e] = 0.f;
          p.lse32[ri] = -INFINITY;
        } else {
          for (int e = 0; e < D; ++e) orow[e] = __float2bfloat16_rn(0.f);
        }
      }
      it = nxt;
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

// Number of SMs of the current device (cached per device).
static int prefill_sms() {
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

template <int D, bool HALF, bool FP8, bool TWO>
cudaError_t launch_prefill_t(const Problem& p, const CUtensorMap& q_map, const CUtensorMap& k_map,
                             const CUtensorMap& v_map,
                             unsigned grid) {
  using C = PrefillCfg<D, FP8 && D == 128>;
  auto k = prefill_kernel<D, HALF, FP8, TWO>;
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, k);
  if (e != cudaSuccess) return e;
  // The register split must fit in what the CTA is launched with.
  if (static_cast<long long>(attr.numRegs) * PF_THREADS < SPLIT_REGS_TOTAL)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // Scores are scaled to log2 units by sl2 = scale * log2(e) (times the K
  // scale of an e4m3 cache).  It is kept strictly positive so a masked score
  // (-inf) always maps to exp2(-inf) = 0; at scale == 0 the visible scores
  // become ~1e-30 * q.k, whose exp2 is 1.0f exactly (uniform weights, as the
  // definition gives).  out_scale is the V scale of an e4m3 cache.
  const float sl2 = fmaxf(p.scale * LOG2E * (FP8 ? p.k_scale : 1.f), 1e-30f);
  const float out_scale = FP8 ? p.v_scale : 1.f;
  k<<<grid, PF_THREADS, C::SMEM, p.stream>>>(p, q_map, k_map, v_map, sl2, out_scale);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const Problem& p, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map) {
  const int NP = (p.G % 2 == 0) ? p.H / 2 : p.H;
  // Persistent grid: one CTA per SM (the shared memory and the 512 TMEM
  // columns of one CTA fill an SM), capped by the host-side bound on items.
  const long long items = static_cast<long long>(p.max_tiles) * NP * p.kv_chunks;
  if (items == 0) return cudaSuccess;
  const unsigned g = static_cast<unsigned>(std::min<long long>(items, prefill_sms()));
  // A 16-bit cache takes two MMA issuers (measured against one: varlen prefill
  // 1.279 -> 1.199 ms, the mixed chunked-prefill step 1.149 -> 1.108 ms).
  if (p.kv_dtype == PATTN_KV_F16)
    return p.D == 128 ? launch_prefill_t<128, true, false, true>(p, q_map, k_map, v_map, g)
                      : launch_prefill_t<64, true, false, true>(p, q_map, k_map, v_map, g);
  // An e4m3 cache at d 128 takes two as well (no warp widens K tiles there:
  // the score MMAs read the codes as they are); at d 64 one.
  if (p.kv_dtype == PATTN_KV_FP8_E4M3)
    return p.D == 128 ? launch_prefill_t<128, false, true, true>(p, q_map, k_map, v_map, g)
                      : launch_prefill_t<64, false, true, false>(p, q_map, k_map, v_map, g);
  return p.D == 128 ? launch_prefill_t<128, false, false, true>(p, q_map, k_map, v_map, g)
                    : launch_prefill_t<64, false, false, true>(p, q_map, k_map, v_map, g);
}

}  // namespace pattn
