// Device helpers shared by the librlk kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rlk {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Hardware base-2 exponential (PTX ex2.approx.ftz.f32; relative error ~2^-22).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch.  A kernel launched after another on the same
// stream with the programmatic-serialization attribute may start while the
// other is still running: pdl_wait() returns once that grid has completed and
// its memory is visible (at once when there is no such grid), so it comes
// before the first read of the other's outputs.  pdl_trigger() lets the next
// such kernel be scheduled once every CTA of this grid has issued it or ended.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// bf16 halves of a 32-bit word as fp32 (exact widening).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_val(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
// A word of two bf16 as a float2 (low half first) / as a bf16 pair.
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ __nv_bfloat162 bf2(uint32_t w) { return *reinterpret_cast<__nv_bfloat162*>(&w); }

// Order-preserving 16-bit key of a bf16 bit pattern: key(a) < key(b) iff a < b
// as numbers; -0 gets the key of +0, so equal values always tie.
__device__ __forceinline__ uint32_t okey16(uint32_t b) {
  b &= 0xFFFFu;
  if (b == 0x8000u) b = 0u;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}
__device__ __forceinline__ uint32_t okey16_inverse(uint32_t k) {
  return (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
}
// Same for fp32 bit patterns (32-bit key).
__device__ __forceinline__ uint32_t okey32(uint32_t b) {
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ uint32_t okey32_inverse(uint32_t k) {
  return (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
}

// ---- double-float (hi + lo) arithmetic, error-free transforms in fp32 ----
struct DF {
  float hi, lo;
};

// Knuth's TwoSum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bp = __fsub_rn(s, a);
  float ap = __fsub_rn(s, bp);
  e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  float hi = __fadd_rn(s, e);
  return DF{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

__device__ __forceinline__ DF df_add_f(DF a, float b) {
  float s, e;
  two_sum(a.hi, b, s, e);
  e = __fadd_rn(e, a.lo);
  float hi = __fadd_rn(s, e);
  return DF{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

// a >= b for normalised double-floats.
__device__ __forceinline__ bool df_ge(DF a, DF b) {
  return (a.hi > b.hi) || (a.hi == b.hi && a.lo >= b.lo);
}

// (a - b) rounded to fp32 (a, b normalised; used for small differences).
__device__ __forceinline__ float df_sub_to_f(DF a, DF b) {
  float s, e;
  two_sum(a.hi, -b.hi, s, e);
  return __fadd_rn(s, __fadd_rn(e, __fsub_rn(a.lo, b.lo)));
}

// p * Z as a double-float (FMA-based exact product of the high parts).
__device__ __forceinline__ DF df_mul_f(DF z, float p) {
  float hi = __fmul_rn(p, z.hi);
  float lo = __fmaf_rn(p, z.hi, -hi);
  lo = __fmaf_rn(p, z.lo, lo);
  float s = __fadd_rn(hi, lo);
  return DF{s, __fsub_rn(lo, __fsub_rn(s, hi))};
}

// ---- mbarrier and bulk-copy wrappers (shared-memory addresses are 32-bit) ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}
// Waits for the phase with the given parity; gives up (returning false and
// raising *abort) after about 2^31 clock cycles, or when *abort is raised.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > (1ll << 31)) {
      *abort = 1;
      return false;
    }
  }
}
// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy ones (a bulk copy into a buffer that was just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Waits for the mbarrier phase of the given parity, suspending in hardware
// (up to ~1 ms a try) rather than polling; gives up (returning false and
// raising *abort) after about 2^31 clock cycles, or when *abort is raised.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, volatile int* abort) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(1000000u)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (clock64() - t0 > (1ll << 31)) {
      *abort = 1;
      return false;
    }
  }
}

// One-dimensional bulk copy global -> shared, completing on an mbarrier
// (addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ float shfl_down(float v, int d) {
  return __shfl_down_sync(0xFFFFFFFFu, v, d);
}
__device__ __forceinline__ float shfl_up(float v, int d) {
  return __shfl_up_sync(0xFFFFFFFFu, v, d);
}

}  // namespace rlk
