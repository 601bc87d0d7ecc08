// dc_device.cuh -- small device helpers for the copy and fold kernels:
// 16-byte loads and stores with explicit cache hints, the byte realignment
// of two aligned 16-byte source blocks, and BF16 <-> binary32 conversion.
#pragma once

#include <stdint.h>

namespace dc {

// ------------------------------------------------------ bounds checks ---
// Built with -DDC_DEBUG_BOUNDS (the checked library, libdc_bounds.so), every
// global load, store and L2 prefetch of the kernels is first checked against
// the range its job allows: for a load or prefetch the 16-byte-block hull of
// the source it reads (a realigning copy reads whole aligned blocks around an
// unaligned span), for a store the exact output range.  An access outside is
// skipped, never made, and the first one is recorded in a device word of its
// translation unit, which dc_check_device reads, clears and reports as
// DC_ERR_BOUNDS; the kernel never traps.  In the normal build every check is
// the constant true and compiles to nothing.
struct BoundsFault {
  unsigned int count;  // accesses outside their range since the last read
  unsigned int site;   // where the first one was (kSite* of its file)
  unsigned long long addr, len, lo, hi;
};
#ifdef DC_DEBUG_BOUNDS
static __device__ BoundsFault g_bounds_fault;
#endif

// True if [a, a + len) lies in [lo, hi); else (checked build) records it.
__device__ __forceinline__ bool in_bounds(const void* a, uint64_t len, uint64_t lo, uint64_t hi,
                                          uint32_t site) {
#ifdef DC_DEBUG_BOUNDS
  const uint64_t x = reinterpret_cast<uint64_t>(a);
  if (x >= lo && x <= hi && len <= hi - x) return true;
  if (atomicAdd(&g_bounds_fault.count, 1u) == 0u) {
    g_bounds_fault.site = site;
    g_bounds_fault.addr = x;
    g_bounds_fault.len = len;
    g_bounds_fault.lo = lo;
    g_bounds_fault.hi = hi;
    __threadfence();
  }
  return false;
#else
  (void)a, (void)len, (void)lo, (void)hi, (void)site;
  return true;
#endif
}

// Defines `cudaError_t NAME(BoundsFault*)`, the host reader of this file's
// record (synchronises the device, reads, clears).
#ifdef DC_DEBUG_BOUNDS
#define DC_BOUNDS_READER(NAME)                                                   \
  cudaError_t NAME(BoundsFault* f) {                                             \
    *f = BoundsFault{};                                                          \
    cudaError_t e = cudaDeviceSynchronize();                                     \
    if (e != cudaSuccess) return e;                                              \
    e = cudaMemcpyFromSymbol(f, g_bounds_fault, sizeof(BoundsFault));            \
    if (e != cudaSuccess || f->count == 0) return e;                             \
    const BoundsFault zero{};                                                    \
    return cudaMemcpyToSymbol(g_bounds_fault, &zero, sizeof(BoundsFault));       \
  }
#else
#define DC_BOUNDS_READER(NAME)   \
  cudaError_t NAME(BoundsFault* f) { \
    *f = BoundsFault{};          \
    return cudaSuccess;          \
  }
#endif

// The 16-byte-block hull of [a, a + n): [hull_lo(a), hull_hi(a, n)).
__host__ __device__ __forceinline__ uint64_t hull_lo(uint64_t a) { return a & ~static_cast<uint64_t>(15); }
__host__ __device__ __forceinline__ uint64_t hull_hi(uint64_t a, uint64_t n) {
  return (a + n + 15) & ~static_cast<uint64_t>(15);
}

// Programmatic dependent launch.  When a kernel is launched with
// programmatic stream serialization, the GPU may start it before the previous
// kernel in the stream has finished; griddepcontrol.wait then blocks until
// that kernel has completed and its writes are visible, so every global
// access below it sees the finished predecessor.  Without that launch
// attribute the wait returns at once.  launch_dependents lets the next
// kernel in the stream (if it was launched the same way) start its launch
// while this one runs; it still waits for this one to finish.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The two halves of pdl_enter, for kernels that do something before the wait.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Bulk prefetch of [p, p + bytes) from HBM into L2 (p 16-byte aligned, bytes a
// multiple of 16).  It moves data between HBM and L2 only; L2 is where every
// SM's loads and stores meet, so a later load still sees any store made in
// between, and the prefetch may be issued before griddepcontrol.wait.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

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

// Coherent 16-byte load that allocates in L1: the realigning reductions read
// every aligned input block twice (the high half of one unit, the low half
// of the next) and may run in place.
__device__ __forceinline__ uint4 ld_cached(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
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

// Output bytes [s, s+16) of the 32-byte little-endian sequence lo || hi
// (s in 0..15): the 32-bit words starting at word s/4 of the sequence, each
// shifted right by 8*(s%4) bits with the next word's low bytes funnelled in.
__device__ __forceinline__ uint4 realign16(const uint4& lo, const uint4& hi, uint32_t s) {
  const uint32_t t = (s & 3u) * 8u;
  uint32_t w0, w1, w2, w3, w4;
  switch (s >> 2) {
    case 0: w0 = lo.x; w1 = lo.y; w2 = lo.z; w3 = lo.w; w4 = hi.x; break;
    case 1: w0 = lo.y; w1 = lo.z; w2 = lo.w; w3 = hi.x; w4 = hi.y; break;
    case 2: w0 = lo.z; w1 = lo.w; w2 = hi.x; w3 = hi.y; w4 = hi.z; break;
    default: w0 = lo.w; w1 = hi.x; w2 = hi.y; w3 = hi.z; w4 = hi.w; break;
  }
  uint4 r;
  r.x = __funnelshift_r(w0, w1, t);
  r.y = __funnelshift_r(w1, w2, t);
  r.z = __funnelshift_r(w2, w3, t);
  r.w = __funnelshift_r(w3, w4, t);
  return r;
}

// The same bytes, the five words picked by two levels of selects (on s & 8,
// then s & 4) instead of a four-way switch.  The gather kernels use this
// form: measured on GB300, 20 calls back to back, payloads at +1 B and the
// output at +3 B, 8 x (1 MiB+1) 3.92 -> 3.77 us and 8 x (4 MiB+1) 12.6 ->
// 12.5 us.  In the FP32 reduction kernels it made ptxas spill registers, so
// those keep realign16.
__device__ __forceinline__ uint4 realign16_sel(const uint4& lo, const uint4& hi, uint32_t s) {
  const uint32_t t = (s & 3u) * 8u;
  const bool h2 = (s & 8u) != 0, h1 = (s & 4u) != 0;
  const uint32_t a0 = h2 ? lo.z : lo.x, a1 = h2 ? lo.w : lo.y, a2 = h2 ? hi.x : lo.z;
  const uint32_t a3 = h2 ? hi.y : lo.w, a4 = h2 ? hi.z : hi.x, a5 = h2 ? hi.w : hi.y;
  const uint32_t w0 = h1 ? a1 : a0, w1 = h1 ? a2 : a1, w2 = h1 ? a3 : a2, w3 = h1 ? a4 : a3,
                 w4 = h1 ? a5 : a4;
  uint4 r;
  r.x = __funnelshift_r(w0, w1, t);
  r.y = __funnelshift_r(w1, w2, t);
  r.z = __funnelshift_r(w2, w3, t);
  r.w = __funnelshift_r(w3, w4, t);
  return r;
}

// Asynchronous 16-byte copy global -> shared (cp.async, cached in L2 only).
// The data travels without passing through registers; the issuing thread
// waits for its own copies with cp.async.wait_group, a hardware wait.
__device__ __forceinline__ void cp_async16(uint32_t smem_addr, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr), "l"(gmem) : "memory");
}
// The same through L1 (.ca): a block that neighbouring threads both copy is
// fetched from L2 once.
__device__ __forceinline__ void cp_async16_ca(uint32_t smem_addr, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_addr), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 ld_shared16(uint32_t smem_addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr)
               : "memory");
  return v;
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

// binary16 <-> binary32 (cvt: the widening is exact; the narrowing rounds to
// nearest even and keeps binary16 subnormals).
__device__ __forceinline__ float f16_to_f32(uint16_t h) {
  float r;
  asm("cvt.f32.f16 %0, %1;" : "=f"(r) : "h"(h));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_f16_rn(float x) {
  uint16_t r;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

}  // namespace dc
