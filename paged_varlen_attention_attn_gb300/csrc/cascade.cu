// cascade.cu -- cascade attention: a common prefix attended once (sm_103a).
//
// "[vLLM] FlashAttention", Cascade Attention (and the use_cascade /
// common_prefix_len fields of FlashAttentionMetadata): when every request of
// a batch starts with the same cached prefix, the prefix attention is
// computed once for all query tokens of the batch -- one request of
// num_tokens queries over common_prefix_len keys, not causal, because every
// query sits after the prefix -- and each request's own suffix (its keys
// past the prefix, causal) separately; the two partial results are merged
// by log-sum-exp.  The result equals plain attention over the whole
// sequence; the prefix's K/V pages are read once for the batch instead of
// once per request.
//
// This file holds the two small kernels around the passes (which reuse the
// prefill and decode kernels in their partial-result mode): the set-up of
// the passes' metadata and the final merge.
#include "../../include/pattn.h"
#include "common.cuh"
#include "internal.h"

namespace pattn {
namespace {

// One CTA: clears the status word, then writes the prefix pass's metadata
// (one request spanning every query token, seq_len = prefix) and each
// request's suffix length.  A suffix shorter than its query (the request's
// cached context does not cover the prefix) is caught as bad metadata by the
// suffix pass's own checks.
__global__ void __launch_bounds__(256)
    cascade_setup_kernel(WsHeader* hdr, const int* qsl, const int* seq_lens, int B, int prefix,
                         int* pre_qsl, int* pre_sl, int* suf_sl) {
  if (threadIdx.x == 0) {
    hdr->status = 0u;
    pre_qsl[0] = qsl[0];
    pre_qsl[1] = qsl[B];
    pre_sl[0] = prefix;
  }
  for (int r = threadIdx.x; r < B; r += blockDim.x) suf_sl[r] = seq_lens[r] - prefix;
}

// One warp per (token, head) row of the batch: out = sum_i 2^(l_i - M) o_i /
// sum_i 2^(l_i - M) over the prefix pass's KA key chunks and the suffix
// pass, l_i their log2-domain lse, M the largest; a partial that saw no key
// (lse = -inf) weighs 0.  A head's attention sink, if any, adds its term to
// the denominator here, once (the passes' partials leave it out).  Rows of
// tokens outside [qsl[0], qsl[B]) are left untouched.
template <int D, bool HALF>
__global__ void __launch_bounds__(256)
    cascade_merge_kernel(const float* o_a, const float* lse_a, int KA, const float* o_b,
                         const float* lse_b, void* out, const int* qsl, int B, int T, int H,
                         const float* sinks) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(T) * H) return;
  const int t = static_cast<int>(row / H);
  if (t < qsl[0] || t >= qsl[B]) return;
  const float b = lse_b[row];
  float M = b;
  for (int c = 0; c < KA; ++c) M = fmaxf(M, lse_a[row * KA + c]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  constexpr int PER = D / 32;
  float acc[PER];
  const int64_t e0 = row * D + lane * PER;
  const float wb = (b == -INFINITY) ? 0.f : exp2f(b - Mu);
  float L = wb;
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = wb * o_b[e0 + e];
  for (int c = 0; c < KA; ++c) {
    const float a = lse_a[row * KA + c];
    if (a == -INFINITY) continue;
    const float wa = exp2f(a - Mu);
    L += wa;
    const float* src = o_a + (row * KA + c) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += wa * src[e];
  }
  L += sink_term(sinks, static_cast<int>(row % H), Mu);
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *(static_cast<unsigned*>(out) + (e0 + e) / 2) = pack2<HALF>(acc[e] * inv, acc[e + 1] * inv);
}

}  // namespace

cudaError_t launch_cascade_setup(WsHeader* hdr, const int* qsl, const int* seq_lens, int B,
                                 int prefix, int* pre_qsl, int* pre_sl, int* suf_sl,
                                 cudaStream_t stream) {
  cascade_setup_kernel<<<1, 256, 0, stream>>>(hdr, qsl, seq_lens, B, prefix, pre_qsl, pre_sl,
                                             suf_sl);
  return cudaGetLastError();
}

cudaError_t launch_cascade_merge(const float* o_a, const float* lse_a, int chunks_a,
                                 const float* o_b, const float* lse_b, void* out, const int* qsl,
                                 int B, int T, int H, int D, bool half, const float* sinks,
                                 cudaStream_t stream) {
  const long long rows = static_cast<long long>(T) * H;
  if (rows == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  if (D == 128) {
    if (half)
      cascade_merge_kernel<128, true><<<grid, 256, 0, stream>>>(o_a, lse_a, chunks_a, o_b, lse_b, out, qsl, B, T, H, sinks);
    else
      cascade_merge_kernel<128, false><<<grid, 256, 0, stream>>>(o_a, lse_a, chunks_a, o_b, lse_b, out, qsl, B, T, H, sinks);
  } else {
    if (half)
      cascade_merge_kernel<64, true><<<grid, 256, 0, stream>>>(o_a, lse_a, chunks_a, o_b, lse_b, out, qsl, B, T, H, sinks);
    else
      cascade_merge_kernel<64, false><<<grid, 256, 0, stream>>>(o_a, lse_a, chunks_a, o_b, lse_b, out, qsl, B, T, H, sinks);
  }
  return cudaGetLastError();
}

}  // namespace pattn
