// dc_device.cuh -- small device helpers for the copy and fold kernels:
// 16-byte loads and stores with explicit cache hints, the byte realignment
// of two aligned 16-byte source blocks, and BF16 <-> binary32 conversion.
#pragma once

#include <stdint.h>

namespace dc {

// Streaming 16-byte load through the read-only path without allocating in
// L1: each source byte of an aligned copy is read exactly once.  Only for
// data that no thread writes during the launch (gather sources).
__device__ __forceinline__ uint4 ld_nc_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Read-only 16-byte load that does allocate in L1: the realigning copy reads
// every aligned source block twice (as the high half of one output vector and
// the low half of the next), and the second read should hit L1.
__device__ __forceinline__ uint4 ld_nc_cached(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Coherent 16-byte load without L1 allocation.  The reductions may run in
// place (an output buffer that is also an input), so they do not use the
// non-coherent read-only path.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st16(uint4* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
               :
               : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Output bytes [s, s+16) of the 32-byte little-endian sequence lo || hi,
// where s = 4*Q + t/8 (t in {0, 8, 16, 24}).  Word j of the result is the
// 32-bit window starting t bits into word Q+j of the sequence.
template <int Q>
__device__ __forceinline__ uint4 realign16(const uint4& lo, const uint4& hi, uint32_t t) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint4 r;
  r.x = __funnelshift_r(w[Q + 0], w[Q + 1], t);
  r.y = __funnelshift_r(w[Q + 1], w[Q + 2], t);
  r.z = __funnelshift_r(w[Q + 2], w[Q + 3], t);
  r.w = __funnelshift_r(w[Q + 3], w[Q + 4], t);
  return r;
}

// BF16 -> binary32 is exact: the 16 bits become the high half of the word.
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two binary32 values -> two BF16 values, each rounded to nearest even, packed
// with `lo` in the low half (the element at the lower address).
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

}  // namespace dc
