// Inline-PTX building blocks for the tensor-memory (tcgen05) decode kernel:
// shared-memory matrix descriptors, the instruction descriptor of
// kind::f8f6f4 MMAs, TMEM allocation, MMA issue and completion, TMEM <->
// register moves, cluster launch control (taking over CTAs of the grid that
// have not started) and named barriers.
#pragma once

#include <stdint.h>

#include "pkv_ptx.cuh"

namespace pkv {
namespace tc {

// Shared-memory matrix descriptor of an operand in the canonical layout
// without swizzling: core matrices of 8 rows x 16 bytes, each 128 contiguous
// bytes (K-major: a row is 16 bytes of K; MN-major: 16 bytes of M or N);
// `lbo` = bytes between core matrices adjacent along K, `sbo` = bytes
// between core matrices adjacent along M or N, for either major-ness.
// Bits 46-48 hold the fixed value 0b001; base offset, stride mode and swizzle
// are 0.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  return d;
}

// Operand formats of kind::f8f6f4.
constexpr uint32_t kFmtE4M3 = 0, kFmtE5M2 = 1;

// Instruction descriptor of a dense kind::f8f6f4 MMA with an fp32
// accumulator: A / B formats, B's major-ness (A is K-major), N and M.
__host__ __device__ constexpr uint32_t idesc_f8f6f4(uint32_t a_fmt, uint32_t b_fmt, bool b_mn_major,
                                                    int n, int m) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// ------------------------------------------------------------------ TMEM --

// Allocate `ncols` (a power of two >= 32) columns of tensor memory; the base
// address is written to `slot` in shared memory.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Free what tmem_alloc allocated.  Whole warp (the allocating one).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Order tcgen05 operations around thread synchronisation.
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread t gets lane (base + t),
// register j column (base + j).
__device__ __forceinline__ void ld_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void st_x16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------- cluster launch control --

// Ask the hardware to cancel the launch of a CTA of this grid that has not
// started yet; the 16-byte answer lands in `resp` (completion on `bar`, 16
// tx bytes).  Issued by one thread.
__device__ __forceinline__ void clc_try_cancel(void *resp, uint64_t *bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128"
      " [%0], [%1];" ::"r"(smem_addr(resp)),
      "r"(smem_addr(bar))
      : "memory");
}

// Read an answer of clc_try_cancel: `ok` = a launch was cancelled, and then
// (x, y, z) is that CTA's index, whose work the caller takes over.
__device__ __forceinline__ void clc_read(const void *resp, uint32_t &ok, uint32_t &x, uint32_t &y,
                                         uint32_t &z) {
  asm volatile(
      "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\tld.shared.b128 r, [%4];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t"
      "clusterlaunchcontrol.query_cancel.get_first_ctaid::y.b32.b128 %2, r;\n\t"
      "clusterlaunchcontrol.query_cancel.get_first_ctaid::z.b32.b128 %3, r;\n\t}"
      : "=r"(ok), "=r"(x), "=r"(y), "=r"(z)
      : "r"(smem_addr(resp))
      : "memory");
}

// --------------------------------------------------------------- misc ----

// Barrier `id` (1..15) among `n` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Two floats -> two E4M3 codes (round to nearest even, saturating to the
// largest finite value): `lo` in bits 0-7, `hi` in bits 8-15.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (bits 0-7, 8-15) -> their values.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t c) {
  uint32_t h2;
  asm("{\n\t.reg .b16 l;\n\tcvt.u16.u32 l, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}"
      : "=r"(h2)
      : "r"(c));
  return __half22float2(*reinterpret_cast<__half2 *>(&h2));
}

}  // namespace tc
}  // namespace pkv
