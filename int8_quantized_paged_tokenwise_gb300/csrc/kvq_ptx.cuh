// Inline-PTX building blocks for the sm_103a kernels: mbarriers with bounded
// waits, TMA (tensor-tiled and 1-D bulk) copies into shared memory, ldmatrix,
// legacy-warp MMA (m16n8k16, FP32 accumulate) and a few bit tricks.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kvq {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------- programmatic dependent launch ---
// Allow the next kernel in the stream (launched with programmatic stream
// serialization) to be scheduled before this grid completes.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the grids this one depends on have completed and their memory
// operations are visible (returns at once without such a dependency).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// try_wait that may suspend the thread for up to `hint_ns` before returning
// false (instead of the system-dependent default), so that a waiting warp
// does not spin on the issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2, %3;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of the barrier to complete, giving up after about
// `limit_ns` nanoseconds of wall time.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------------------ TMA ---
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// The same copy with an L2 evict-first policy: for data read once per call
// (the K/V pages of a decode), so that its lines are the first to go instead
// of lines other kernels still use or have yet to write back.
__device__ __forceinline__ void tma_load_2d_evict_first(uint32_t dst, const CUtensorMap* map,
                                                        int32_t x, int32_t y, uint32_t bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}

// 1-D bulk copy; dst, src 16-byte aligned and bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bulk prefetch of global memory into L2 (no shared-memory destination);
// src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 8-byte shared load that the compiler may not hoist out of a loop (keeps
// loop-invariant operands in shared memory instead of registers).
__device__ __forceinline__ uint2 lds_u2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// ------------------------------------------------------------ ldmatrix ---
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// ----------------------------------------------------------------- MMA ---
// D(16x8, f32) = A(16x16) * B(16x8) + C; only the rows g (not g+8) of C/D
// are carried: the caller's upper 8 rows of A are zero (padded query heads).
template <bool BF16>
__device__ __forceinline__ void mma_16816(float& d0, float& d1, uint32_t a0, uint32_t a2,
                                          uint32_t b0, uint32_t b1) {
  float x2, x3;
  const float z = 0.f;
  const uint32_t zr = 0u;
  if constexpr (BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d0), "=f"(d1), "=f"(x2), "=f"(x3)
        : "r"(a0), "r"(zr), "r"(a2), "r"(zr), "r"(b0), "r"(b1), "f"(d0), "f"(d1), "f"(z), "f"(z));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d0), "=f"(d1), "=f"(x2), "=f"(x3)
        : "r"(a0), "r"(zr), "r"(a2), "r"(zr), "r"(b0), "r"(b1), "f"(d0), "f"(d1), "f"(z), "f"(z));
  }
}

// D(16x8, f32) += A(16x16) * B(16x8), all four accumulator registers live:
// d[0] = (row g, col 2c), d[1] = (g, 2c+1), d[2] = (g+8, 2c), d[3] = (g+8, 2c+1).
template <bool BF16>
__device__ __forceinline__ void mma_16816_acc(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  if constexpr (BF16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Transpose of an 8x8 matrix of 16-bit elements held as an MMA fragment
// (thread (g, c) holds row g, columns 2c and 2c+1) within the warp.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Largest of the 32 lanes' values (every lane gets it).
__device__ __forceinline__ uint32_t redux_max_u32(uint32_t x) {
  uint32_t y;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(y) : "r"(x));
  return y;
}

// ------------------------------------------------------------ numerics ---
// The largest of three floats in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^e as a float, for e in [-126, 127] (exact; built from the exponent field).
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// Power-of-two exponent that brings a set of BF16 values into FP16's normal
// range without loss: given the largest magnitude's bit pattern (sign
// cleared), the shift sh such that that magnitude times 2^-sh lies in
// [2^14, 2^15); sh is kept in [-126, 113] so that 2^sh and 2^-sh are normal
// floats.  A zero (or subnormal) maximum gives -126.
__device__ __forceinline__ int bf16_fp16_shift(uint32_t max_bits) {
  const int eb = (int)(max_bits >> 7);          // biased BF16 exponent, 0..255
  const int sh = eb - 127 - 14;
  return sh < -126 ? -126 : (sh > 113 ? 113 : sh);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) {
  return *reinterpret_cast<__half2*>(&u);
}
__device__ __forceinline__ uint32_t bf2_as_u32(__nv_bfloat162 h) {
  return *reinterpret_cast<uint32_t*>(&h);
}

// Four packed int8 codes -> two packed FP16 pairs, exactly.  After flipping
// the sign bit each byte u = code + 128 is placed under the exponent byte
// 0x64, giving the FP16 value 1024 + u; subtracting 1152 leaves the code.
// `sel_lo`/`sel_hi` choose which two bytes form each pair.
template <uint32_t SEL_LO, uint32_t SEL_HI>
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
  lo = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, SEL_LO)), bias));
  hi = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, SEL_HI)), bias));
}

// The same without the subtraction: each FP16 value is 1152 + code, exactly.
// Used where the bias is removed after the MMA (a dot product with such a row
// is the dot product with the codes plus 1152 times the sum of the other
// operand).
template <uint32_t SEL_LO, uint32_t SEL_HI>
__device__ __forceinline__ void i8x4_to_h2x2_b1152(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, SEL_LO);
  hi = __byte_perm(u, 0x64646464u, SEL_HI);
}

}  // namespace kvq
