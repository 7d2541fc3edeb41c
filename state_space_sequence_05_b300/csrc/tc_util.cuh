// tc_util.cuh -- device helpers shared by the tensor-core forward kernels:
// bounded mbarrier waits, acquire/release flags, special-function-unit
// exponentials and the bf16 hi/lo operand split.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "tc_ptx.cuh"

namespace ssd {
namespace tc {

// Default bound on one wait: 2 s of global time.
constexpr unsigned long long kWaitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded mbarrier wait: true once the phase with parity `parity` has
// completed, false after `limit_ns` of global time.  Each probe may suspend
// the thread until the barrier changes; the clock is read only every 32
// probes, so a waiting warp costs few issue slots.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity,
                                         unsigned long long limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = gtime();
#pragma unroll 1
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 31u) == 0 && gtime() - t0 > limit_ns) return false;
  }
}

// Warp-collective form: every lane waits and the warp agrees on the result,
// so a timeout never splits a warp (later warp-synchronous instructions
// would otherwise strand the lanes that went on).
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity,
                                              unsigned long long limit_ns = kWaitNs) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, limit_ns));
}

// The math warps meet at `bar` (initialised with their count; phase parity
// `par`); bounded.  They synchronise only through mbarriers so that a
// timed-out warp can leave without stranding the others at a hardware
// barrier.
__device__ __forceinline__ bool math_sync(uint64_t* bar, uint32_t par,
                                          unsigned long long limit_ns = kWaitNs) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  return wait_bar_warp(bar, par, limit_ns);
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 2^x on the special-function unit (ex2.approx.ftz: relative error ~2^-22,
// flushes subnormal results to zero, which every use here tolerates).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2 on the special-function unit (lg2.approx.ftz: absolute error ~2^-22
// near 1)
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
// two floats rounded to bf16 (to nearest, ties to even), a in the low half
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// v ~= hi + lo: hi = v with its low 16 bits cleared (bf16 by truncation),
// lo = v - hi (exact in fp32) truncated to bf16 the same way; |v - hi - lo|
// < 2^-14 |v|.  Packs the hi and lo halves of two values (a in the low 16
// bits, as __floats2bfloat162_rn(a, b) would).
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  hi = __byte_perm(ua, ub, 0x7632);
  const float la = a - __uint_as_float(ua & 0xffff0000u);
  const float lb = b - __uint_as_float(ub & 0xffff0000u);
  lo = __byte_perm(__float_as_uint(la), __float_as_uint(lb), 0x7632);
}

// ---- packed fp32 pairs (the sm_100-family f32x2 instructions: one
// instruction computes both lanes of a pair; each lane rounds as its fp32
// operation would).
struct f2 {
  float x, y;
};
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
  f2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
  f2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// a * b + c, both lanes
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
// split2 on a pair: hi = both values truncated to bf16, lo = the remainders
// truncated the same way (|v - hi - lo| < 2^-14 |v|); x in the low 16 bits.
__device__ __forceinline__ void split2p(f2 v, uint32_t& hi, uint32_t& lo) {
  const uint32_t ua = __float_as_uint(v.x), ub = __float_as_uint(v.y);
  hi = __byte_perm(ua, ub, 0x7632);
  const f2 r = sub2(v, f2{__uint_as_float(ua & 0xffff0000u), __uint_as_float(ub & 0xffff0000u)});
  lo = __byte_perm(__float_as_uint(r.x), __float_as_uint(r.y), 0x7632);
}
// the two bf16 values of a packed word as fp32 (low half first)
__device__ __forceinline__ f2 bf2(uint32_t w) {
  return f2{__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)};
}

}  // namespace tc
}  // namespace ssd
