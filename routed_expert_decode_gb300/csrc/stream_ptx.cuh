// stream_ptx.cuh -- mbarrier and bulk-copy (cp.async.bulk) helpers and the
// 16-byte dp4a chunk dot, shared by the kernels that stream expert weights
// through shared memory (the fused decode kernel and the streamed GEMV).
//
// A stage of shared memory is filled by one-CTA bulk copies (no multicast)
// that complete transaction bytes on the stage's "full" mbarrier; its readers
// arrive on an "empty" mbarrier when done.  Every wait is bounded.
#pragma once

#include "moe_internal.cuh"

namespace moe {

constexpr int kSpinIters = 1 << 26;  // iteration cap of every wait
constexpr int kSuspendNs = 20000;    // mbarrier try_wait suspend-time hint

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// raise the phase's expected transaction bytes without arriving
__device__ __forceinline__ void mbar_add_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// bounded wait for completion of the phase with the given parity.  Each try_wait
// may suspend the thread (up to kSuspendNs) until the phase completes, so a
// waiting warp does not take issue slots from the warps sharing its SM
// sub-partition.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long budget) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  for (int i = 0; i < kSpinIters; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity), "n"(kSuspendNs)
        : "memory");
    if (done) return true;
    if (clock64() - t0 > budget) return false;
  }
  return false;
}

// non-blocking: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// one-CTA bulk copy global -> shared (16-byte aligned addresses, size a
// multiple of 16), completing its bytes on `bar`
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint4 lds16(const int8_t *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

// exact int32 dot of 16 int8 pairs
__device__ __forceinline__ int dot16(const uint4 &a, const uint4 &b) {
  int s = __dp4a((int)a.x, (int)b.x, 0);
  s = __dp4a((int)a.y, (int)b.y, s);
  s = __dp4a((int)a.z, (int)b.z, s);
  return __dp4a((int)a.w, (int)b.w, s);
}

// MOE_FLAG_DEBUG_TAPS: index j of tapped feature n of a row of `width` outputs
// (n == tap_feature(j, width)), or -1
__device__ __forceinline__ int tapped(uint32_t n, uint32_t width) {
  int jt = -1;
#pragma unroll
  for (int j = 0; j < kNTap; ++j)
    if (tap_feature((uint32_t)j, width) == n) jt = j;
  return jt;
}

// the exact int32 dot of a 32-block whose two 16-byte halves lanes 2i and 2i+1
// hold (chunk counts are even, so both lanes of a pair always run together)
__device__ __forceinline__ int pair_sum(int v, int lane) {
  return v + __shfl_xor_sync(3u << (lane & 30), v, 1);
}

}  // namespace moe
