// plan.cu -- per-call work list, built on the device so the host never waits.
//
// The FA3 backend of "[vLLM] FlashAttention" (AOT scheduling section)
// computes the distribution of work before the attention kernel runs; this is
// the same idea with a layout of our own: one CTA reads query_start_loc and
// seq_lens, validates them, and writes the prefill tiles (request, 128-row
// query-row item) ordered by their number of key tiles, largest first, so the
// heaviest tiles start first (longest-processing-time order).  It also clears
// the status word, so later kernels of the same call report into a clean one,
// and the decode kernel's partition counters.
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

__global__ void __launch_bounds__(PLAN_THREADS) plan_kernel(const Problem p) {
  __shared__ int hist[NBUCKET];
  __shared__ int warp_sums[PLAN_THREADS / 32];
  const int tid = threadIdx.x;
  if (tid == 0 && p.clear_status) p.hdr->status = 0u;
  for (int i = tid; i < p.B * p.Hkv; i += PLAN_THREADS) p.counters[i] = 0u;
  for (int b = tid; b < NBUCKET; b += PLAN_THREADS) hist[b] = 0;
  __syncthreads();

  // Pass 1: validate requests, histogram prefill tiles by cost.
  for (int r = tid; r < p.B; r += PLAN_THREADS) {
    int q_len, s, t0;
    if (!request_ok(p, r, q_len, s, t0)) {
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
    for (int qt = 0; qt < nt; ++qt) atomicAdd(&hist[tile_cost(p, q_len, s, qt)], 1);
  }
  __syncthreads();

  // Exclusive scan over buckets in descending cost order: bucket b starts at
  // the number of tiles with a larger cost.  Each thread owns 4 buckets.
  constexpr int PER = NBUCKET / PLAN_THREADS;
  int local[PER];
  int sum = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int b = NBUCKET - 1 - (tid * PER + e);
    local[e] = hist[b];
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
    int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_sums[lane] = wi - w;  // exclusive prefix of warps
  }
  __syncthreads();
  int run = warp_sums[wid] + incl - sum;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int b = NBUCKET - 1 - (tid * PER + e);
    const int c = local[e];
    hist[b] = run;  // cursor: first slot of bucket b
    run += c;
  }
  if (tid == PLAN_THREADS - 1) {
    if (run > p.max_tiles) flag_status(&p.hdr->status, PATTN_DEV_BAD_METADATA);
    p.hdr->num_prefill_tiles = min(run, p.max_tiles);
  }
  __syncthreads();

  // Pass 2: scatter (request, q-tile) pairs to their slots.
  for (int r = tid; r < p.B; r += PLAN_THREADS) {
    int q_len, s, t0;
    if (!request_ok(p, r, q_len, s, t0) || q_len <= 1) continue;
    const int nt = (q_len + p.rows_per_item - 1) / p.rows_per_item;
    for (int qt = 0; qt < nt; ++qt) {
      const int slot = atomicAdd(&hist[tile_cost(p, q_len, s, qt)], 1);
      if (slot < p.max_tiles) p.tiles[slot] = make_int2(r, qt);
    }
  }
}

// Decode-only calls: clear the status word and the partition counters.  The
// decode kernel follows as a programmatic dependent, so it starts streaming the
// cache while this runs and waits for it only where it touches these words.
__global__ void __launch_bounds__(PLAN_THREADS) decode_prep_kernel(unsigned* words, int n) {
  grid_dep_trigger();
  for (int i = threadIdx.x; i < n; i += blockDim.x) words[i] = 0u;
}

}  // namespace

cudaError_t launch_plan(const Problem& p) {
  plan_kernel<<<1, PLAN_THREADS, 0, p.stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_prep(void* ws, size_t bytes, cudaStream_t stream) {
  const int n = static_cast<int>(bytes / sizeof(unsigned));
  decode_prep_kernel<<<1, PLAN_THREADS, 0, stream>>>(static_cast<unsigned*>(ws), n);
  return cudaGetLastError();
}

}  // namespace pattn
