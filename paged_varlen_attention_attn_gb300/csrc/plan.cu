// plan.cu -- per-call work list, built on the device so the host never waits.
//
// The FA3 backend of "[vLLM] FlashAttention" (AOT scheduling section)
// computes the distribution of work before the attention kernel runs; this is
// the same idea with a layout of our own: one CTA reads query_start_loc and
// seq_lens, validates them, and writes the prefill tiles (request, 128-row
// query-row item) ordered by their number of key tiles, largest first, so the
// heaviest tiles start first (longest-processing-time order).  It also clears
// the status word, so later kernels of the same call report into a clean one,
// and the decode kernel's partition counters, and orders the decode requests
// by their visible length, longest first, for the decode grid.
#include "../../include/pattn.h"
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

constexpr int PLAN_THREADS = 1024;
constexpr int NBUCKET = 4096;  // cost buckets (key tiles); larger costs share the last

__device__ __forceinline__ bool request_ok(const Problem& p, int r, int& q_len, int& s, int& t0) {
  t0 = p.qsl[r];
  q_len = p.qsl[r + 1] - t0;
  s = p.seq_lens[r];
  return q_len >= 0 && (q_len <= s || p.long_queries) && s <= p.mbps * p.bs && t0 >= 0 &&
         t0 + q_len <= p.T;
}

__device__ __forceinline__ int tile_cost(const Problem& p, int q_len, int s, int qt) {
  const int ctx = s - q_len;
  const int i0 = qt * p.rows_per_item;
  const int i_last = min(q_len, i0 + p.rows_per_item) - 1;
  const int lo = (p.window > 0) ? max(0, ctx + i0 - p.window + 1) : 0;
  const int hi = p.causal ? min(s, ctx + i_last + 1) : s;
  const int c = (hi + BLOCK_N - 1) / BLOCK_N - lo / BLOCK_N;
  return min(max(c, 0), NBUCKET - 1);
}

// Visible KV blocks of a request's decode row (its partitions' total work), or
// 0 for a request that is not a valid decode (it does no decode work).
__device__ __forceinline__ int decode_cost_of(const Problem& p, int q_len, int s) {
  if (q_len != 1 || s < 1 || s > p.mbps * p.bs) return 0;
  const int k_lo = (p.window > 0) ? max(0, s - p.window) : 0;
  return min((s + p.bs - 1) / p.bs - k_lo / p.bs, NBUCKET - 1);
}
__device__ __forceinline__ int decode_cost(const Problem& p, int r) {
  return decode_cost_of(p, p.qsl[r + 1] - p.qsl[r], p.seq_lens[r]);
}

// Turns hist[] (counts per cost bucket) into cursors in descending cost
// order: bucket b starts at the number of items with a larger cost.  Returns
// the total count (in every thread).  Each thread owns NBUCKET / PLAN_THREADS
// buckets; warp_sums has a slot per warp.
__device__ int scan_descending(int* hist, int* warp_sums) {
  constexpr int PER = NBUCKET / PLAN_THREADS;
  const int tid = threadIdx.x;
  int local[PER];
  int sum = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    local[e] = hist[NBUCKET - 1 - (tid * PER + e)];
    sum += local[e];
  }
  int incl = sum;
  const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_sums[lane] = wi - w;  // exclusive prefix of warps
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  int run = warp_sums[wid] + incl - sum;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    hist[NBUCKET - 1 - (tid * PER + e)] = run;  // cursor: first slot of the bucket
    run += local[e];
  }
  const int total = warp_sums[32];
  __syncthreads();
  return total;
}

// Adds n to hist[key] for every lane in `lanes` (the calling lanes, which
// all execute this) and returns each lane's old value plus its rank among the
// lanes with the same key: one shared-memory atomic per distinct key in the
// warp (decode batches often share one cost, whose lane-by-lane atomics
// would serialise).
__device__ __forceinline__ int hist_add_warp(int* hist, int key, unsigned lanes) {
  const int lane = threadIdx.x & 31;
  const unsigned peers = __match_any_sync(lanes, key);
  const int leader = __ffs(peers) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(&hist[key], __popc(peers));
  base = __shfl_sync(peers, base, leader);
  return base + __popc(peers & ((1u << lane) - 1u));
}

// Writes p.decode_order: every request, by decreasing decode cost (a counting
// sort; the order within one cost is whatever the atomics give).  cost0 is
// the decode cost of the thread's first request (request tid), which the
// caller read; a larger batch reads the rest here.  Adds the visible KV
// blocks of every decode row to *blocks.  The whole warp walks the requests
// together (its lanes past the batch take no part), so that its atomics can
// be combined.
__device__ void order_decodes(const Problem& p, int* hist, int* warp_sums,
                              unsigned long long* blocks, int cost0) {
  const int tid = threadIdx.x, lane = tid & 31;
  for (int b = tid; b < NBUCKET; b += PLAN_THREADS) hist[b] = 0;
  __syncthreads();
  for (int r = tid; r - lane < p.B; r += PLAN_THREADS) {
    const bool in = r < p.B;
    const unsigned lanes = __ballot_sync(0xffffffffu, in);
    const int c = !in ? 0 : (r == tid ? cost0 : decode_cost(p, r));
    if (in) hist_add_warp(hist, c, lanes);
    const unsigned sum = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(c));
    if (lane == 0) atomicAdd(blocks, static_cast<unsigned long long>(sum));
  }
  __syncthreads();
  scan_descending(hist, warp_sums);
  for (int r = tid; r - lane < p.B; r += PLAN_THREADS) {
    const bool in = r < p.B;
    const unsigned lanes = __ballot_sync(0xffffffffu, in);
    if (in) p.decode_order[hist_add_warp(hist, r == tid ? cost0 : decode_cost(p, r), lanes)] = r;
  }
}

// Estimated time (us) of a mixed batch whose prefill keeps `gs` SMs and
// whose decode runs on the other `m` = num_sms - gs at the same time, then on
// every SM once prefill is done.  Prefill: the longest-processing-time list is
// walked in rounds of gs items, a round lasting about its first (largest)
// item, and never less than the total work over gs SMs.  Decode: m SMs
// stream at dec_bytes_per_us each, capped by the HBM bandwidth beside prefill.
// cost[t]: the key tiles of sorted tile t (kept in shared memory by pass 2).
// (fp32 throughout: an estimate, and GB300's fp64 is slow)
__device__ float co_schedule_estimate(const Problem& p, const unsigned short* cost, int gs,
                                      int n_items, int np, float work_items, float dec_bytes) {
  float rounds = 0.f;
  for (int x = 0; x < n_items; x += gs) rounds += static_cast<float>(cost[x / np]);
  const float t_pre = p.pf_us_per_tile * fmaxf(rounds, work_items / gs);
  const int m = p.num_sms - gs;
  const float full_rate = fminf(p.num_sms * p.dec_bytes_per_us, p.hbm_bytes_per_us);
  if (m <= 0) return t_pre + dec_bytes / full_rate;
  const float rate = fminf(m * p.dec_bytes_per_us, p.hbm_bytes_per_us);
  const float t_dec = dec_bytes / rate;
  if (t_dec <= t_pre) return t_pre;
  return t_pre + (dec_bytes - rate * t_pre) / full_rate;
}

__global__ void __launch_bounds__(PLAN_THREADS) plan_kernel(const Problem p) {
  __shared__ int hist[NBUCKET];
  __shared__ int warp_sums[PLAN_THREADS / 32 + 1];
  __shared__ unsigned long long s_tile_work, s_dec_blocks;
  __shared__ float s_best[PLAN_THREADS / 32];
  __shared__ int s_best_gs[PLAN_THREADS / 32];
  __shared__ unsigned short s_cost[NBUCKET];  // cost of sorted tile t < NBUCKET
  const int tid = threadIdx.x;
  // Request tid's metadata is read once, here, and kept in registers for
  // every pass (a batch of more than PLAN_THREADS requests reads the others
  // in each pass).
  int q_len0 = 0, s0 = 0, t00 = 0;
  const bool ok0 = tid < p.B && request_ok(p, tid, q_len0, s0, t00);
  if (tid == 0) {
    s_tile_work = 0ull;
    s_dec_blocks = 0ull;
  }
  if (tid == 0 && p.clear_status) p.hdr->status = 0u;
  if (tid == 0) p.hdr->next_item = 0u;
  for (int i = tid; i < p.B * p.Hkv; i += PLAN_THREADS) p.counters[i] = 0u;
  for (int b = tid; b < NBUCKET; b += PLAN_THREADS) hist[b] = 0;
  __syncthreads();

  // Pass 1: validate requests, histogram prefill tiles by cost.
  for (int r = tid; r < p.B; r += PLAN_THREADS) {
    int q_len = q_len0, s = s0, t0 = t00;
    if (r == tid ? !ok0 : !request_ok(p, r, q_len, s, t0)) {
      flag_status(&p.hdr->status, PATTN_DEV_BAD_METADATA);
      // Rows of a bad prefill request are written as zeros (decode rows are
      // handled by the decode kernel), clamped to the output buffer.
      if (q_len > 1) {
        const int a = max(0, t0), b = min(p.T, t0 + q_len);
        const int64_t e0 = static_cast<int64_t>(a) * p.H * p.D, e1 = static_cast<int64_t>(b) * p.H * p.D;
        if (p.o32) {
          for (int64_t e = e0; e < e1; ++e) p.o32[e] = 0.f;
          for (int64_t e = static_cast<int64_t>(a) * p.H; e < static_cast<int64_t>(b) * p.H; ++e)
            p.lse32[e] = -INFINITY;
        } else {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
          for (int64_t e = e0; e < e1; ++e) out[e] = __float2bfloat16_rn(0.f);
        }
      }
      continue;
    }
    if (q_len <= 1) continue;
    const int nt = (q_len + p.rows_per_item - 1) / p.rows_per_item;
    unsigned long long work = 0ull;
    for (int qt = 0; qt < nt; ++qt) {
      const int c = tile_cost(p, q_len, s, qt);
      atomicAdd(&hist[c], 1);
      work += static_cast<unsigned long long>(c);
    }
    atomicAdd(&s_tile_work, work);
  }
  __syncthreads();

  // Bucket b's tiles start at the number of tiles with a larger cost.
  const int run = scan_descending(hist, warp_sums);
  if (tid == 0) {
    if (run > p.max_tiles) flag_status(&p.hdr->status, PATTN_DEV_BAD_METADATA);
    p.hdr->num_prefill_tiles = min(run, p.max_tiles);
  }

  // Pass 2: scatter (request, q-tile) pairs to their slots.
  for (int r = tid; r < p.B; r += PLAN_THREADS) {
    int q_len = q_len0, s = s0, t0 = t00;
    if ((r == tid ? !ok0 : !request_ok(p, r, q_len, s, t0)) || q_len <= 1) continue;
    const int nt = (q_len + p.rows_per_item - 1) / p.rows_per_item;
    for (int qt = 0; qt < nt; ++qt) {
      const int c = tile_cost(p, q_len, s, qt);
      const int slot = atomicAdd(&hist[c], 1);
      if (slot < p.max_tiles) p.tiles[slot] = make_int2(r, qt);
      if (slot < NBUCKET) s_cost[slot] = static_cast<unsigned short>(c);
    }
  }
  __syncthreads();

  // Pass 3: the decode grid's request order.
  if (p.decode_order)
    order_decodes(p, hist, warp_sums, &s_dec_blocks,
                  tid < p.B ? decode_cost_of(p, q_len0, s0) : 0);
  __syncthreads();

  // Pass 4 (mixed batches): how many SMs the prefill kernel keeps.  Each
  // thread estimates a few prefill grid sizes; the fastest estimate wins (the
  // largest grid on ties).
  if (!p.co_schedule) {
    if (tid == 0) p.hdr->prefill_ctas = 0;
    return;
  }
  const int np = ((p.G % 2) == 0 ? p.H / 2 : p.H) * p.kv_chunks;
  const int n_items = min(run, p.max_tiles) * np;  // (run: every thread has it)
  const float dec_bytes = static_cast<float>(s_dec_blocks) * static_cast<float>(p.bs * p.Hkv) *
                          2.f * p.D * (p.kv_dtype == PATTN_KV_FP8_E4M3 ? 1.f : 2.f);
  const float work_items = static_cast<float>(s_tile_work) * np;
  float best = INFINITY;
  int best_gs = p.num_sms;
  // (the tile costs are kept for the first NBUCKET sorted tiles; a batch with
  // more keeps every SM for its prefill)
  if (n_items > 0 && dec_bytes > 0.f && n_items / np <= NBUCKET) {
    for (int gs = p.num_sms - tid; gs >= max(1, p.num_sms / 2); gs -= PLAN_THREADS) {
      const float e = co_schedule_estimate(p, s_cost, gs, n_items, np, work_items, dec_bytes);
      if (e < best || (e == best && gs > best_gs)) {
        best = e;
        best_gs = gs;
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int og = __shfl_xor_sync(0xffffffffu, best_gs, o);
    if (ob < best || (ob == best && og > best_gs)) {
      best = ob;
      best_gs = og;
    }
  }
  if ((tid & 31) == 0) {
    s_best[tid >> 5] = best;
    s_best_gs[tid >> 5] = best_gs;
  }
  __syncthreads();
  if (tid == 0) {
    float b = s_best[0];
    int g = s_best_gs[0];
    for (int w = 1; w < PLAN_THREADS / 32; ++w)
      if (s_best[w] < b || (s_best[w] == b && s_best_gs[w] > g)) {
        b = s_best[w];
        g = s_best_gs[w];
      }
    p.hdr->prefill_ctas = (b == INFINITY) ? 0 : g;
  }
}

// Decode-only calls: clear the status word and the partition counters and
// write the decode order.  The decode kernel follows as a programmatic
// dependent: its CTAs are resident when this finishes, which saves the launch
// gap.
__global__ void __launch_bounds__(PLAN_THREADS) decode_prep_kernel(const Problem p) {
  __shared__ int hist[NBUCKET];
  __shared__ int warp_sums[PLAN_THREADS / 32 + 1];
  __shared__ unsigned long long s_dec_blocks;
  grid_dep_trigger();
  if (threadIdx.x == 0) {
    p.hdr->status = 0u;
    p.hdr->num_prefill_tiles = 0;
    p.hdr->prefill_ctas = 0;
    p.hdr->next_item = 0u;
    s_dec_blocks = 0ull;
  }
  for (int i = threadIdx.x; i < p.B * p.Hkv; i += PLAN_THREADS) p.counters[i] = 0u;
  order_decodes(p, hist, warp_sums, &s_dec_blocks,
                threadIdx.x < p.B ? decode_cost(p, threadIdx.x) : 0);
}

}  // namespace

cudaError_t launch_plan(const Problem& p) {
  plan_kernel<<<1, PLAN_THREADS, 0, p.stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_prep(const Problem& p) {
  decode_prep_kernel<<<1, PLAN_THREADS, 0, p.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pattn
