// Shared device helpers for the thinmx kernels (sm_103a).
//
// Everything here is inline PTX or plain CUDA C++ written for this library:
// mbarrier + bulk-copy (TMA 1D) staging, programmatic dependent launch,
// bounded waits, E2M1 decode and mixed-precision FMA.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tt {

// ---------------------------------------------------------------------------
// Error reporting from device code.  Kernels get a pointer to the library's
// device error word; the first error code written wins.
// ---------------------------------------------------------------------------
constexpr int kErrNull = 1;     // TT_ERR_NULL
constexpr int kErrAlign = 3;    // TT_ERR_ALIGN
constexpr int kErrNonfinite = 4;  // TT_ERR_NONFINITE
constexpr int kErrTimeout = 7;  // TT_ERR_TIMEOUT

__device__ __forceinline__ void flag_error(int32_t* word, int code) {
  if (word) atomicCAS(word, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A bounded wait gives up after this long (the copies it waits on take
// microseconds; a second means something is broken).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers and bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_inval(uint32_t bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking: true if the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps (up to `hint_ns`)
// until the phase completes instead of spinning and taking issue slots from
// the warps that have work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Suspend-time hint of the bounded wait (0: plain try_wait).  try_wait
// already suspends the thread until the phase completes or a hardware time
// limit passes (measured: polls that come back unsatisfied are rare), so
// neither a hint, a back-off between polls nor a non-blocking poll loop
// changed the time or the instruction count.
#ifndef TT_WAIT_HINT_NS
#define TT_WAIT_HINT_NS 0
#endif

// Waits for the phase with the given parity to complete; false if it did not
// within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (TT_WAIT_HINT_NS > 0 ? mbar_try_wait_sleep(bar, parity, TT_WAIT_HINT_NS)
                            : mbar_try_wait(bar, parity))
      return true;
    if ((it & 15u) == 0u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// L2 policy for small data that later calls read again (activations).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ld_global_v4_hint(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// L2 policy for data read exactly once (streamed weights).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Global -> shared bulk copy (TMA, non-tensor).  dst, src 16-byte aligned,
// bytes a multiple of 16.  Completion is signalled as tx bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Global -> L2 bulk prefetch (no shared-memory destination, no completion
// tracking).  src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Both are no-ops when the kernel was not
// launched with the programmatic-serialization attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Numerics
// ---------------------------------------------------------------------------
// E8M0 byte -> fp32 2^(b-127).  b = 0 gives the subnormal 2^-127 (bit 22);
// b = 255 gives +Inf, which turns the (zero) codes of a NaN block into NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  uint32_t bits = max(b << 23, 0x00400000u);
  return __uint_as_float(bits);
}

// Eight E2M1 codes (one 32-bit word, code for even k in the low nibble of
// each byte) -> four f16x2 values, the even-k value in the low half.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& h0, uint32_t& h1,
                                                uint32_t& h2, uint32_t& h3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

// acc_lo += lo(a) * lo(b); acc_hi += hi(a) * hi(b).  f16 x f16 products are
// exact in fp32, so each step rounds once, in fp32.
__device__ __forceinline__ void fma_f16x2_f32(float& acc_lo, float& acc_hi, uint32_t a,
                                              uint32_t b) {
  asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "mov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %1, ah, bh, %1;\n\t}"
      : "+f"(acc_lo), "+f"(acc_hi)
      : "r"(a), "r"(b));
}

// Same with bf16 operands (bf16 x bf16 is exact in fp32).
__device__ __forceinline__ void fma_bf16x2_f32(float& acc_lo, float& acc_hi, uint32_t a,
                                               uint32_t b) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "mov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.bf16 %1, ah, bh, %1;\n\t}"
      : "+f"(acc_lo), "+f"(acc_hi)
      : "r"(a), "r"(b));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// Power-of-two exponent s such that m * 2^s lies in [2^14, 2^15) for the
// largest magnitude m (> 0, finite); 0 when m is 0 or not finite.
__device__ __forceinline__ int f16_prescale_exponent(float m) {
  uint32_t bits = __float_as_uint(m);
  int e = int((bits >> 23) & 0xFF);
  if (e == 0 || e == 255) return 0;  // zero/subnormal max, or non-finite
  return 14 - (e - 127);
}

// x * 2^s rounded to f16 (exact for the bf16 inputs that stay >= 2^-14).
__device__ __forceinline__ uint32_t pack_f16x2_scaled(float a, float b, float two_s) {
  __half2 h = __floats2half2_rn(a * two_s, b * two_s);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + expf(-g)) * u;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sums a (lanes 0..15 get the total) and b (lanes 16..31 get the total) over
// the warp with five shuffles.
__device__ __forceinline__ float warp_sum2(float a, float b, int lane) {
  const bool lo = lane < 16;
  float keep = lo ? a : b;
  float send = lo ? b : a;
  keep += __shfl_xor_sync(0xffffffffu, send, 16);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
  return keep;
}

}  // namespace tt
