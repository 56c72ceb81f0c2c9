// common.cuh -- device helpers shared by the kernels of libpattn (sm_103a).
//
// Hand-written inline PTX for the Blackwell data movers and tensor cores:
// mbarrier, TMA (cp.async.bulk.tensor), cp.async, ldmatrix / mma.sync, and
// tcgen05 (TMEM alloc, MMA, commit, ld/st).  Every spin wait is bounded: it
// gives up after PATTN_WAIT_LIMIT_NS of %globaltimer, records
// PATTN_DEV_TIMEOUT in the status word, and returns false so the caller can
// unwind.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pattn {

// Device status bits, OR-ed into the workspace status word.
constexpr unsigned PATTN_DEV_BAD_METADATA = 1u;
constexpr unsigned PATTN_DEV_TIMEOUT = 2u;

// A wait that has not finished after this long is treated as a hang.  The
// wait-test build (PATTN_WAIT_TEST, a separate library that only the tests
// load) shortens it so that a test can make a wait run out quickly.
#ifdef PATTN_WAIT_TEST
constexpr unsigned long long PATTN_WAIT_LIMIT_NS = 10000000ull;  // 10 ms
#else
constexpr unsigned long long PATTN_WAIT_LIMIT_NS = 2000000000ull;  // 2 s
#endif

constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void flag_status(unsigned* status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned bar_addr, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// flags PATTN_DEV_TIMEOUT, and sets *abort) if it does not within the limit
// or if another role already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, unsigned* status,
                                          volatile int* abort_flag) {
  const unsigned a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(a, parity)) return true;
    if (abort_flag && *abort_flag) return false;
    if (globaltimer_ns() - t0 > PATTN_WAIT_LIMIT_NS) {
      flag_status(status, PATTN_DEV_TIMEOUT);
      if (abort_flag) *abort_flag = 1;
      return false;
    }
  }
}

// After a role gave up on a wait, a producer waits (bounded, whatever the
// abort flag says) for the copies it armed on the stages of a ring of nst
// stages, so that no copy is still writing shared memory when the CTA frees
// its resources and exits.  Ring positions [0, armed_end) were armed in
// order, position j on barrier bars[j % nst] in phase j / nst; the latest
// position of each stage is the only phase of that barrier that can still be
// open, and earlier phases of the same stage completed before it was armed.
// skip_pos is a position that was not armed (-1: none).
__device__ __forceinline__ void drain_armed(uint64_t* bars, int nst, int armed_end, int skip_pos,
                                            unsigned* status) {
  for (int j = armed_end - nst; j < armed_end; ++j) {
    if (j < 0 || j == skip_pos) continue;
    mbar_wait(&bars[j % nst], (j / nst) & 1, status, nullptr);
  }
}

// ------------------------------------------------------------ attention sinks

// The normaliser term of head h's attention sink against a row whose
// log2-domain reference max is M: 2^(sink_h * log2(e) - M), or 0 without a
// sink (a null array or a sink of -inf).  A sink far above M gives +inf, which
// drives the row to 0, its limit.
__device__ __forceinline__ float sink_term(const float* sinks, int h, float M) {
  if (sinks == nullptr) return 0.f;
  const float s2 = sinks[h] * 1.4426950408889634f;
  return (s2 == -INFINITY) ? 0.f : exp2f(s2 - M);
}

// ------------------------------------------------- programmatic dependent launch

// Block until the kernel this one depends on (launched before it in the
// stream) has finished and its writes are visible; a no-op without a
// programmatic dependency.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the dependent kernel to launch once every CTA of this grid has executed
// this (or exited).
__device__ __forceinline__ void grid_dep_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "r"(c4)
      : "memory");
}

// Named barrier over `count` threads (a multiple of 32) of the CTA; id 0 is
// the one __syncthreads uses.
__device__ __forceinline__ void named_bar_sync(unsigned id, unsigned count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy
// (TMA, tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- cp.async

__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------- ldmatrix / mma.sync

__device__ __forceinline__ void ldsm_x4(unsigned addr, unsigned& r0, unsigned& r1, unsigned& r2,
                                        unsigned& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(unsigned addr, unsigned& r0, unsigned& r1,
                                          unsigned& r2, unsigned& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, fp32 accumulate.
// D += A B on e4m3 operands: m16n8k32, A 16 x 32 row-major (four registers of
// four codes), B 32 x 8 column-major (two registers), fp32 accumulation.
__device__ __forceinline__ void mma_16832_e4m3(float (&d)[4], unsigned a0, unsigned a1,
                                               unsigned a2, unsigned a3, unsigned b0,
                                               unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 codes (the low 16 bits of v) -> f16x2, exactly (the hardware pair
// conversion; every e4m3 value is an f16 value).
__device__ __forceinline__ unsigned e4m3x2_to_f16x2(unsigned v) {
  unsigned r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<unsigned short>(v)));
  return r;
}

// f16x2 -> two e4m3 codes (low half -> low byte), round to nearest, saturating.
__device__ __forceinline__ unsigned f16x2_to_e4m3x2(unsigned h) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}

// A bf16 pair (w), times sc = 2^k, as e4m3 hi and lo codes with hi + lo equal
// to the scaled pair: hi rounds the 8-bit significand to 4 bits, and the
// remainder (at most 4 significant bits, exact in f16) is lo.  Exact while the
// scaled value's remainder is no finer than e4m3's smallest step (2^-9).
__device__ __forceinline__ void split_pair(unsigned w, float sc, unsigned& hi, unsigned& lo) {
  const __half2 y = __floats2half2_rn(__uint_as_float(w << 16) * sc,
                                      __uint_as_float(w & 0xffff0000u) * sc);
  const unsigned yb = *reinterpret_cast<const unsigned*>(&y);
  hi = f16x2_to_e4m3x2(yb);
  const unsigned hb = e4m3x2_to_f16x2(hi);
  const __half2 r = __hsub2(y, *reinterpret_cast<const __half2*>(&hb));
  lo = f16x2_to_e4m3x2(*reinterpret_cast<const unsigned*>(&r));
}

// The power of two 2^k that puts a bf16 magnitude with exponent field eb in
// [2^7, 2^8) (k clamped to +-126), and its inverse.
__device__ __forceinline__ void split_scale(int eb, float& sc, float& inv) {
  const int k = min(126, max(-126, 134 - eb));
  sc = __int_as_float((k + 127) << 23);
  inv = __int_as_float((127 - k) << 23);
}

template <bool F16>
__device__ __forceinline__ void mma_16816(float (&d)[4], unsigned a0, unsigned a1, unsigned a2,
                                          unsigned a3, unsigned b0, unsigned b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

template <bool F16>
__device__ __forceinline__ unsigned pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<unsigned*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<unsigned*>(&h);
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(unsigned* dst_smem, unsigned ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(unsigned taddr, unsigned ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One MMA, both operands from shared memory descriptors.
__device__ __forceinline__ void tc_mma_ss(unsigned d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          unsigned idesc, unsigned accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with 8-bit operands (kind::f8f6f4: K = 32 per MMA; both e4m3 with
// an instruction descriptor whose A and B type fields are 0).
__device__ __forceinline__ void tc_mma_ss_f8(unsigned d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             unsigned idesc, unsigned accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// One MMA, A from tensor memory, B from a shared memory descriptor.
__device__ __forceinline__ void tc_mma_ts(unsigned d_tmem, unsigned a_tmem, uint64_t b_desc,
                                          unsigned idesc, unsigned accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on bar once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld32(unsigned taddr, float (&v)[32]) {
  unsigned* r = reinterpret_cast<unsigned*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tc_st32(unsigned taddr, const float (&v)[32]) {
  const unsigned* r = reinterpret_cast<const unsigned*>(v);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 16 packed 32-bit columns (e.g. 32 bf16 values) into this thread's lane.
__device__ __forceinline__ void tc_st16u(unsigned taddr, const unsigned (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// Shared memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (16-byte units), descriptor version 1 at bit 46,
// swizzle mode in bits 61..63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(unsigned saddr, unsigned lbo_bytes,
                                                    unsigned sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
//   ab_bf16: A and B are bf16 (else f16); b_mn_major: B is MN-major.
__host__ __device__ constexpr unsigned make_idesc_f16(int M, int N, bool ab_bf16,
                                                      bool b_mn_major) {
  return (1u << 4)                                   // D: f32
         | ((ab_bf16 ? 1u : 0u) << 7)                // A type
         | ((ab_bf16 ? 1u : 0u) << 10)               // B type
         | ((b_mn_major ? 1u : 0u) << 16)            // B major
         | (static_cast<unsigned>(N >> 3) << 17)     // N / 8
         | (static_cast<unsigned>(M >> 4) << 24);    // M / 16
}

}  // namespace pattn
