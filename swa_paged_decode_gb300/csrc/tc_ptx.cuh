// tc_ptx.cuh -- thin inline-PTX wrappers for the sm_103a tensor-core path:
// mbarriers, TMEM allocation, tcgen05.mma / commit / ld / st, shared-memory
// matrix descriptors and the fp8 / fp4 -> f16 conversions.
#pragma once

#include <stdint.h>

namespace dsa {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of a phase (mbarrier.try_wait may suspend the thread
// until the phase completes or a hardware time limit passes; test_wait
// returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait whose budget is exact in SM cycles: polls without suspending.
__device__ __forceinline__ bool mbar_wait_strict(uint64_t *bar, uint32_t parity, long long budget) {
  const long long t0 = clock64();
  while (!mbar_test_wait(bar, parity))
    if (clock64() - t0 > budget) return false;
  return true;
}
// try_wait that lets the thread sleep (up to `ns` nanoseconds, woken early
// when the phase completes) instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait on a phase: gives up (returns false) after `budget` SM
// clock cycles. With `sleep_ns` > 0 the thread sleeps between polls (woken
// early when the phase completes), leaving issue slots to busy warps.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long budget,
                                          uint32_t sleep_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!(sleep_ns ? mbar_try_wait_sleep(bar, parity, sleep_ns) : mbar_try_wait(bar, parity)))
    if (clock64() - t0 > budget) return false;
  return true;
}

// Shared-memory add with acquire-release order at CTA scope (the writes
// that precede it in this thread are visible to the thread that observes
// its result, and vice versa); returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel_shared(uint32_t *a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_u32(a)), "r"(v)
               : "memory");
  return old;
}

// ------------------------------------------------------------ fences
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------ TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 lanes x 32 bit, N consecutive columns -> N registers per thread; the
// wait is inside the same statement so the outputs are ready on return.
#define DSA_TMEM_LD8(taddr, r)                                                              \
  asm volatile(                                                                             \
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"        \
      "tcgen05.wait::ld.sync.aligned;"                                                      \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), \
        "=r"(r[7])                                                                          \
      : "r"(taddr)                                                                          \
      : "memory")

#define DSA_TMEM_ST8(taddr, r)                                                             \
  asm volatile(                                                                            \
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"       \
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),                                       \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]) \
      : "memory")

// x16 load without the wait; pair with tmem_wait16 on the same registers
// (the wait names them, so no use can move above it).
#define DSA_TMEM_LD16_NOWAIT(taddr, r)                                                    \
  asm volatile(                                                                           \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "                                           \
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"                   \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),           \
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),         \
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])                                \
      : "r"(taddr)                                                                        \
      : "memory")

// Waits for every outstanding tcgen05.ld of the warp; the 32 registers are
// tied to the wait so their uses stay below it.
#define DSA_TMEM_WAIT32(a, b)                                                             \
  asm volatile("tcgen05.wait::ld.sync.aligned;"                                           \
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),  \
                 "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), \
                 "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]),          \
                 "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),  \
                 "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]),            \
                 "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15])                       \
               :                                                                          \
               : "memory")

// Two x16 loads (columns c0.. and c1..) under one wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, uint32_t (&a)[16],
                                            uint32_t (&b)[16]) {
  DSA_TMEM_LD16_NOWAIT(ta, a);
  DSA_TMEM_LD16_NOWAIT(tb, b);
  DSA_TMEM_WAIT32(a, b);
}

// Register budget of a warpgroup (multiple of 8); the four warps of the
// warpgroup execute it together.
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// N columns in groups of 8.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float *v) {
#pragma unroll
  for (int g = 0; g < N / 8; ++g) {
    uint32_t r[8];
    DSA_TMEM_LD8(taddr + 8 * g, r);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[8 * g + i] = __uint_as_float(r[i]);
  }
}
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float *v) {
#pragma unroll
  for (int g = 0; g < N / 8; ++g) {
    uint32_t r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(v[8 * g + i]);
    DSA_TMEM_ST8(taddr + 8 * g, r);
  }
}

// ------------------------------------------------------------ MMA
// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), version 1, swizzle mode.
enum : uint32_t { kSwzNone = 0, kSwz128 = 2, kSwz64 = 4, kSwz32 = 6 };
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                          uint32_t swz) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swz << 61);
}

// Instruction descriptor, kind::f16: D f32, A and B f16, dense.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// No "memory" clobber: the MMA touches shared memory and TMEM only through
// the async proxy, ordered by the fences and barriers around it (all volatile
// asm, which the compiler keeps in program order); a clobber here would force
// reloads of spilled values before every MMA.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
// Arrive on `bar` once every tcgen05 op this thread issued so far completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------ conversions
// Four e4m3 codes (byte i = element i) -> two f16x2 words (exact).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// Two e4m3 codes in the low 16 bits -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w16) {
  uint32_t r;
  asm("{\n\t.reg .b16 a, b;\n\t"
      "mov.b32 {a, b}, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\t}"
      : "=r"(r)
      : "r"(w16));
  return r;
}
// Eight e2m1 nibbles (byte i holds elements 2i (low) and 2i+1 (high)) ->
// four f16x2 words (exact).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 32-byte load (sm_100+): one request per 32-byte sector; p 32-byte aligned.
__device__ __forceinline__ void ldg_nc_v8(const void *p, uint4 &a, uint4 &b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                 "=r"(b.w)
               : "l"(p));
}

// Bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) into L2 by the
// TMA engine: no registers, no L1 miss tracking.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void *p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// Read-only 16-byte load kept in L1, issued where it stands (volatile: not
// merged with or hoisted above another load of the same address, so the
// value need not stay in registers between uses).
__device__ __forceinline__ float4 ldg_f4_here(const float4 *p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace tc
}  // namespace dsa
