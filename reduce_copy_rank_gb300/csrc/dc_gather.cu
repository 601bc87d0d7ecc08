// dc_gather.cu -- the rank-ordered all-gather copy (copy_rank_ordered).
//
// "perf(cuda): vectorize the deterministic all-gather copy and right-size its
// single-block path" (RL-Kernel PR 491), section "What": the gathered output
// is the concatenation of the P payloads in rank order, byte for byte.  When
// the output, the size and every payload are 16-byte aligned, one flat loop
// over all ranks' 16-byte vectors keeps every thread busy across ranks;
// otherwise each rank is copied with vectors where possible and bytes at the
// edges.  The same page names the old defect this design avoids: one byte per
// thread and a 64-bit division per byte to find the source rank.
//
// Design on one GB300:
//  * The unit of work is a 16-byte-aligned OUTPUT vector.  A launch covers
//    the output vectors of one or more jobs (all_gather_many packs several
//    gathers into one launch), numbered by a prefix over the jobs.  Each CTA
//    owns one contiguous run of them, so no thread ever searches for its rank
//    per element: the CTA finds its first job and rank once (one 64-bit
//    division per CTA and job), then walks ranks in order.
//  * Aligned job (flat): rank r owns output vectors [r*B/16, (r+1)*B/16); all
//    threads of a CTA stream each rank's part of its run with LDG.128 /
//    STG.128, UNROLL vectors in flight per thread.
//  * Unaligned job: the vectors that lie inside one rank's bytes are
//    "interior"; their source starts at a fixed offset s = (src - dst) mod 16.
//    For s = 0 they are copied like the flat case; otherwise each output
//    vector is built from the two aligned source blocks that cover it with a
//    funnel shift, so loads and stores both stay 16 bytes wide and aligned.
//    The few vectors that mix two ranks' bytes (one per rank boundary) or
//    stick out of the output (first and last) are written byte by byte by one
//    warp.  Reads never leave the 16-byte blocks that hold source bytes, so
//    they stay inside the source allocation.
//  * Jobs with fewer than kGatherSmallBytes per rank are copied byte by byte.
#include "dc_device.cuh"
#include "dc_internal.h"

namespace dc {
namespace {

template <int BLOCK, int UNROLL>
__device__ __forceinline__ void copy_aligned(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                             uint32_t n) {
  for (uint32_t i = threadIdx.x; i < n; i += BLOCK * UNROLL) {
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint32_t k = i + u * BLOCK;
      if (k < n) v[u] = ld_nc_stream(src + k);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint32_t k = i + u * BLOCK;
      if (k < n) st16(dst + k, v[u]);
    }
  }
}

// dst[k] = bytes [s, s+16) of src[k] || src[k+1], s = 4*Q + t/8, for k < n.
// Both blocks hold source bytes of output vector k, so they are in bounds.
template <int BLOCK, int UNROLL, int Q>
__device__ __forceinline__ void copy_realign_q(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                               uint32_t n, uint32_t t) {
  for (uint32_t i = threadIdx.x; i < n; i += BLOCK * UNROLL) {
    uint4 lo[UNROLL], hi[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint32_t k = i + u * BLOCK;
      if (k < n) {
        lo[u] = ld_nc_cached(src + k);
        hi[u] = ld_nc_cached(src + k + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint32_t k = i + u * BLOCK;
      if (k < n) st16(dst + k, realign16<Q>(lo[u], hi[u], t));
    }
  }
}

template <int BLOCK>
__device__ __forceinline__ void copy_realign(const uint4* src, uint4* dst, uint32_t n, uint32_t s) {
  constexpr int U = kGatherRealignUnroll;
  const uint32_t t = (s & 3u) * 8u;
  switch (s >> 2) {  // uniform across the CTA
    case 0: copy_realign_q<BLOCK, U, 0>(src, dst, n, t); break;
    case 1: copy_realign_q<BLOCK, U, 1>(src, dst, n, t); break;
    case 2: copy_realign_q<BLOCK, U, 2>(src, dst, n, t); break;
    default: copy_realign_q<BLOCK, U, 3>(src, dst, n, t); break;
  }
}

// Output vectors [k0, k1) of a job that lie inside rank r's bytes
// [d_r, d_r + B); the source of output byte x is src_r + (x - d_r).
template <int BLOCK, int UNROLL>
__device__ __forceinline__ void copy_interior(uint64_t src_r, uint64_t d_r, uint64_t vbase,
                                              uint64_t k0, uint64_t k1) {
  const uint64_t dst_addr = (vbase + k0) << 4;
  const uint64_t src_addr = src_r + (dst_addr - d_r);
  const uint32_t s = static_cast<uint32_t>(src_addr & 15u);
  const uint32_t n = static_cast<uint32_t>(k1 - k0);
  uint4* dst = reinterpret_cast<uint4*>(dst_addr);
  if (s == 0)
    copy_aligned<BLOCK, UNROLL>(reinterpret_cast<const uint4*>(src_addr), dst, n);
  else
    copy_realign<BLOCK>(reinterpret_cast<const uint4*>(src_addr - s), dst, n, s);
}

// One output vector that holds bytes of rank r and possibly rank r+1, or
// bytes outside the job's output (first and last vector): lanes 0..15 of warp
// 0 copy the bytes that belong to the output, one each.
template <int MAXJ, int MAXS>
__device__ __forceinline__ void copy_boundary(const GatherParams<MAXJ, MAXS>& p, const GatherJob& J,
                                              uint64_t vbase, uint64_t k, uint32_t r) {
  const uint32_t lane = threadIdx.x;
  if (lane >= 16) return;
  const uint64_t x = ((vbase + k) << 4) + lane;
  const uint64_t out_end = J.out + static_cast<uint64_t>(p.P) * J.bytes;
  if (x < J.out || x >= out_end) return;
  uint64_t d = J.out + static_cast<uint64_t>(r) * J.bytes;
  uint32_t q = r;
  if (x >= d + J.bytes) {  // B >= kGatherSmallBytes > 16: at most the next rank
    ++q;
    d += J.bytes;
  }
  const uint8_t* src = reinterpret_cast<const uint8_t*>(p.src[J.src0 + q]);
  *reinterpret_cast<uint8_t*>(x) = src[x - d];
}

template <int BLOCK, int UNROLL, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_flat(const GatherParams<MAXJ, MAXS>& p, const GatherJob& J,
                                            uint64_t a, uint64_t b) {
  const uint64_t vp = J.bytes >> 4;  // vectors per rank
  uint64_t r = a / vp;                // once per CTA and job
  uint64_t k = a;
  uint4* out = reinterpret_cast<uint4*>(J.out);
  while (k < b) {
    const uint64_t e = min(b, (r + 1) * vp);
    const uint4* src = reinterpret_cast<const uint4*>(p.src[J.src0 + r]) + (k - r * vp);
    copy_aligned<BLOCK, UNROLL>(src, out + k, static_cast<uint32_t>(e - k));
    k = e;
    ++r;
  }
}

template <int BLOCK, int UNROLL, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_unaligned(const GatherParams<MAXJ, MAXS>& p,
                                                 const GatherJob& J, uint64_t a, uint64_t b) {
  const uint64_t B = J.bytes;
  const uint64_t vbase = J.out >> 4;
  const uint64_t first_byte = max(J.out, (vbase + a) << 4);
  uint32_t r = static_cast<uint32_t>((first_byte - J.out) / B);  // once per CTA and job
  if (a == 0 && (J.out & 15u)) copy_boundary(p, J, vbase, 0, 0);
  for (; r < static_cast<uint32_t>(p.P); ++r) {
    const uint64_t d = J.out + static_cast<uint64_t>(r) * B;
    const uint64_t e = d + B;
    const uint64_t lo = ((d + 15) >> 4) - vbase;  // first vector inside rank r
    const uint64_t hi = (e >> 4) - vbase;         // one past the last one
    if (lo >= b) break;
    const uint64_t ia = max(a, lo), ib = min(b, hi);
    if (ia < ib) copy_interior<BLOCK, UNROLL>(p.src[J.src0 + r], d, vbase, ia, ib);
    if ((e & 15u) && hi >= a && hi < b) copy_boundary(p, J, vbase, hi, r);
  }
}

// Fewer than kGatherSmallBytes per rank: every output byte of the CTA's
// vectors is copied on its own.  P*B < kMaxRanks*kGatherSmallBytes, so the
// rank lookup is a 32-bit division over a few thousand bytes in total.
template <int BLOCK, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_small(const GatherParams<MAXJ, MAXS>& p, const GatherJob& J,
                                             uint64_t a, uint64_t b) {
  const uint64_t vbase = J.out >> 4;
  const uint32_t B = static_cast<uint32_t>(J.bytes);
  const uint32_t total = static_cast<uint32_t>(p.P) * B;
  const uint32_t nbytes = static_cast<uint32_t>(b - a) * 16u;
  const uint64_t x0 = (vbase + a) << 4;
  for (uint32_t i = threadIdx.x; i < nbytes; i += BLOCK) {
    const uint64_t x = x0 + i;
    if (x < J.out) continue;
    const uint32_t off = static_cast<uint32_t>(x - J.out);
    if (off >= total) continue;
    const uint32_t r = off / B;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.src[J.src0 + r]);
    *reinterpret_cast<uint8_t*>(x) = src[off - r * B];
  }
}

template <int BLOCK, int UNROLL, bool FLAT, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_cta(const GatherParams<MAXJ, MAXS>& p, uint64_t g0,
                                           uint64_t g1) {
  int j = 0;
  while (j + 1 < p.njobs && p.job[j].vfirst + p.job[j].nvec <= g0) ++j;
  for (; j < p.njobs && p.job[j].vfirst < g1; ++j) {
    const GatherJob& J = p.job[j];
    const uint64_t a = max(g0, J.vfirst) - J.vfirst;
    const uint64_t b = min(g1, J.vfirst + J.nvec) - J.vfirst;
    if (a >= b) continue;
    if constexpr (FLAT) {
      gather_flat<BLOCK, UNROLL>(p, J, a, b);
    } else {
      if (J.flags & kJobFlat)
        gather_flat<BLOCK, UNROLL>(p, J, a, b);
      else if (J.flags & kJobSmall)
        gather_small<BLOCK>(p, J, a, b);
      else
        gather_unaligned<BLOCK, UNROLL>(p, J, a, b);
    }
  }
}

// Multi-CTA gather: CTA c owns output vectors [c*chunk, (c+1)*chunk).
// FLAT: every job of the launch is 16-byte aligned (the flat path only).
template <int MAXJ, int MAXS, bool FLAT>
__global__ void __launch_bounds__(kGatherBlock)
    dc_gather_kernel(const __grid_constant__ GatherParams<MAXJ, MAXS> p) {
  const uint64_t g0 = static_cast<uint64_t>(blockIdx.x) * p.chunk_vec;
  if (g0 >= p.total_vec) return;
  const uint64_t g1 = min(g0 + p.chunk_vec, p.total_vec);
  gather_cta<kGatherBlock, kGatherUnroll, FLAT>(p, g0, g1);
}

// Single-CTA gather for small outputs: one CTA copies everything.
template <int MAXJ, int MAXS, bool FLAT>
__global__ void __launch_bounds__(FLAT ? kGatherSingleBlock : kGatherSingleBlockGeneral)
    dc_gather_single_kernel(const __grid_constant__ GatherParams<MAXJ, MAXS> p) {
  constexpr int kBlock = FLAT ? kGatherSingleBlock : kGatherSingleBlockGeneral;
  gather_cta<kBlock, kGatherUnroll, FLAT>(p, 0, p.total_vec);
}

template <int MAXJ, int MAXS>
bool all_flat(const GatherParams<MAXJ, MAXS>& p) {
  for (int j = 0; j < p.njobs; ++j)
    if (!(p.job[j].flags & kJobFlat)) return false;
  return true;
}

template <int MAXJ, int MAXS>
cudaError_t launch_impl(const GatherParams<MAXJ, MAXS>& p, int grid, bool single, cudaStream_t s) {
  const bool flat = all_flat(p);
  if (single) {
    if (flat)
      dc_gather_single_kernel<MAXJ, MAXS, true><<<1, kGatherSingleBlock, 0, s>>>(p);
    else
      dc_gather_single_kernel<MAXJ, MAXS, false><<<1, kGatherSingleBlockGeneral, 0, s>>>(p);
  } else {
    if (flat)
      dc_gather_kernel<MAXJ, MAXS, true><<<grid, kGatherBlock, 0, s>>>(p);
    else
      dc_gather_kernel<MAXJ, MAXS, false><<<grid, kGatherBlock, 0, s>>>(p);
  }
  return cudaGetLastError();
}

// Resident CTAs per SM of the general (heavier) instantiation, so a grid
// planned from it never exceeds what either instantiation can hold at once.
template <int MAXJ, int MAXS>
int occupancy_impl() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dc_gather_kernel<MAXJ, MAXS, false>,
                                                    kGatherBlock, 0) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_gather(const GatherParams1& p, int grid, bool single, cudaStream_t s) {
  return launch_impl(p, grid, single, s);
}
cudaError_t launch_gather(const GatherParamsS& p, int grid, bool single, cudaStream_t s) {
  return launch_impl(p, grid, single, s);
}
cudaError_t launch_gather(const GatherParamsL& p, int grid, bool single, cudaStream_t s) {
  return launch_impl(p, grid, single, s);
}

int gather_ctas_per_sm(int which) {
  switch (which) {
    case 0: return occupancy_impl<1, kMaxRanks>();
    case 1: return occupancy_impl<kManySmallTensors, kManySmallSegments>();
    default: return occupancy_impl<kManyMaxTensors, kManyMaxSegments>();
  }
}

}  // namespace dc
