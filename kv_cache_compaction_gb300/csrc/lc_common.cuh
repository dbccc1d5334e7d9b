// Device helpers shared by the compaction kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lc_ptx.cuh"

namespace lc {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kInf = __builtin_huge_valf();

// Per-head status values written by the solver kernels (same numbers as the
// public lc_status codes).
constexpr int LC_OK_STATUS = 0;
constexpr int LC_NOT_CONVERGED_STATUS = 5;
constexpr int LC_SINGULAR_STATUS = 6;

// 2^x via the hardware approximation instruction (flushes subnormal results
// to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// x = hi + lo with hi = fp16(x) and lo = fp16(x - hi): the pair carries about
// 22 significant bits, so products of pairs keep fp32-level accuracy on the
// 16-bit tensor-core path.
__device__ __forceinline__ void split_f16(float x, __half& hi, __half& lo) {
  hi = __float2half_rn(x);
  lo = __float2half_rn(x - __half2float(hi));
}

__device__ __forceinline__ uint32_t pack_h2(__half a, __half b) {
  return static_cast<uint32_t>(__half_as_ushort(a)) |
         (static_cast<uint32_t>(__half_as_ushort(b)) << 16);
}

__device__ __forceinline__ uint32_t f2_to_h2(float a, float b);

// Split 8 floats into two uint4 of packed fp16 (hi parts, lo parts), for
// values in the fp16 range.  hi is x with its mantissa cut to the 10 bits fp16
// stores (a bit mask), so it converts to fp16 exactly and lo = x - hi is exact
// in fp32 with |lo| < 2^-10 |x|; lo rounded to fp16 leaves a relative error
// below 2^-21 in hi + lo.  One mask, one subtraction and one packed
// conversion per element.
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
  float h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    h[i] = __uint_as_float(__float_as_uint(x[i]) & 0xFFFFE000u);
    l[i] = x[i] - h[i];
  }
  hi = make_uint4(f2_to_h2(h[0], h[1]), f2_to_h2(h[2], h[3]), f2_to_h2(h[4], h[5]),
                  f2_to_h2(h[6], h[7]));
  lo = make_uint4(f2_to_h2(l[0], l[1]), f2_to_h2(l[2], l[3]), f2_to_h2(l[4], l[5]),
                  f2_to_h2(l[6], l[7]));
}

__device__ __forceinline__ uint32_t f2_to_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8_f16(const float* x) {
  return make_uint4(f2_to_h2(x[0], x[1]), f2_to_h2(x[2], x[3]), f2_to_h2(x[4], x[5]),
                    f2_to_h2(x[6], x[7]));
}

// Order-preserving map of a non-NaN float to uint32 (larger float -> larger
// code); -0 and +0 map to the same code.
__device__ __forceinline__ uint32_t order_code(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) == 0) b = 0;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float order_decode(uint32_t c) {
  uint32_t b = (c & 0x80000000u) ? (c & 0x7fffffffu) : ~c;
  return __uint_as_float(b);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Bounded mbarrier wait used by the warp-specialised kernels.  Gives up when
// another role of this CTA has aborted (*abort_flag), when any CTA of the
// launch has timed out (timeout bit in the global error word), or after
// kWaitLimitNs; on a timeout it sets both flags so everyone winds down.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((++n & 255u) == 0 && (*reinterpret_cast<volatile uint32_t*>(err) & kErrWaitTimeout)) {
      *abort_flag = 1;
      return false;
    }
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrWaitTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// One 32-bit word of a row of 16-bit elements, folded into a row hash: -0 is
// mapped onto +0 in both halves (so that equal values hash equally), then
// the word is mixed with its position.  A row's hash is the sum of its
// words' mixes.
__device__ __forceinline__ uint32_t row_word_mix(uint32_t x, int pos) {
  if ((x & 0x7fffu) == 0) x &= 0xffff0000u;
  if ((x & 0x7fff0000u) == 0) x &= 0x0000ffffu;
  x ^= 0x9e3779b9u * static_cast<uint32_t>(pos + 1);
  x *= 0x85ebca6bu;
  x ^= x >> 13;
  x *= 0xc2b2ae35u;
  x ^= x >> 16;
  return x;
}

// Bounded wait on the way out of a kernel: returns once the phase of `bar`
// with the given parity has completed, or after kWaitLimitNs; abort flags are
// not consulted (the point is to let work already in flight finish).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

// Run by the thread that issued a kernel's tensor-core operations, after its
// last issue and before the CTA frees its tensor memory: commits every
// operation it issued to `bar` (an mbarrier of count 1 used for nothing else)
// and waits, bounded, for them to complete.  Then no MMA still reads or
// writes tensor or shared memory when the CTA frees them, also when a wait
// elsewhere in the CTA gave up early and the pipeline was abandoned midway.
__device__ __forceinline__ void drain_mma(uint64_t* bar) {
  umma_commit(bar);
  drain_wait(bar, 0);
}

// True if an earlier CTA of this launch (or an earlier launch of this call)
// already timed out.
__device__ __forceinline__ bool launch_aborted(const uint32_t* err) {
  return (*reinterpret_cast<const volatile uint32_t*>(err) & kErrWaitTimeout) != 0;
}

__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

}  // namespace lc
