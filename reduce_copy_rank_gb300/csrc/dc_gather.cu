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
//    owns one contiguous run of them and finds its first job once.
//  * Inside a run, thread t takes vectors t, t+BLOCK, t+2*BLOCK, ..., UNROLL
//    of them at a time with all loads issued before the first store, across
//    rank boundaries: the flat loop of the page.  (The page's first version
//    copied rank by rank, leaving threads idle and serialising the ranks'
//    reads; a per-rank walk inside a CTA has the same defect.)  A thread's
//    vector index only grows, so it finds its rank by walking forward from
//    the rank of the run's first vector: comparisons, never a division per
//    element.
//  * Aligned job (flat): plain LDG.128 / STG.128.
//  * Unaligned job: each output vector that lies inside one rank's bytes is
//    built from the two aligned source blocks that cover it with a funnel
//    shift, so loads and stores stay 16 bytes wide and aligned; the few
//    vectors that straddle two ranks or stick out of the output (at most P+1
//    per job) are written byte by byte.
//  * Jobs with fewer than kGatherSmallBytes per rank are copied byte by byte.
#include "dc_device.cuh"
#include "dc_internal.h"

namespace dc {
namespace {

// Aligned job (flat): rank r owns output vectors [r*vp, (r+1)*vp), vp = B/16.
// Thread t copies vectors a+t, a+t+BLOCK, ... of the CTA's run [a, b), UNROLL
// at a time with every load issued before the first store, so the whole
// CTA's run is in flight at once whatever the rank boundaries.  A thread's
// vector index only grows, so its rank is found by walking forward from the
// rank of the run's first vector: one 64-bit division per thread, then
// comparisons (at most P steps in total).
template <int BLOCK, int UNROLL, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_flat(const GatherParams<MAXJ, MAXS>& p, const GatherJob& J,
                                            uint64_t a, uint64_t b) {
  const uint64_t vp = J.bytes >> 4;
  uint64_t r = a / vp;
  uint64_t rbeg = r * vp, rend = rbeg + vp;
  uint4* out = reinterpret_cast<uint4*>(J.out);
  for (uint64_t i = a + threadIdx.x; i < b; i += static_cast<uint64_t>(BLOCK) * UNROLL) {
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint64_t k = i + static_cast<uint64_t>(u) * BLOCK;
      if (k < b) {
        while (k >= rend) {
          ++r;
          rbeg = rend;
          rend += vp;
        }
        v[u] = ld_nc_stream(reinterpret_cast<const uint4*>(p.src[J.src0 + r]) + (k - rbeg));
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint64_t k = i + static_cast<uint64_t>(u) * BLOCK;
      if (k < b) st16(out + k, v[u]);
    }
  }
}

// Unaligned job (B >= kGatherSmallBytes).  Output vector k covers bytes
// [x, x+16), x = 16*(vbase+k).  It is "interior" when all 16 bytes belong to
// one rank r (d_r <= x and x+16 <= d_r + B): its source starts at
// src_r + (x - d_r), at offset s = that address mod 16, so it is built from
// the aligned source block holding that byte and the next one (one block
// when s = 0) and stored as one aligned 16-byte vector.  The other vectors
// (one per rank boundary, plus the first and last vector when the output is
// not aligned) are written byte by byte by the thread that owns them; since
// B > 16 they hold bytes of at most two ranks.  Both aligned source blocks
// of an interior vector contain bytes of [src_r, src_r + B), so no read
// leaves the 16-byte blocks of the source buffer.  Threads walk ranks
// forward as in the flat case.
template <int BLOCK, int UNROLL, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_unaligned(const GatherParams<MAXJ, MAXS>& p,
                                                 const GatherJob& J, uint64_t a, uint64_t b) {
  const uint64_t B = J.bytes;
  const uint64_t vbase = J.out >> 4;
  const uint64_t out_end = J.out + static_cast<uint64_t>(p.P) * B;
  const uint64_t first_byte = max(J.out, (vbase + a) << 4);
  uint32_t r = static_cast<uint32_t>((first_byte - J.out) / B);
  uint64_t d = J.out + static_cast<uint64_t>(r) * B;  // rank r's first output byte
  uint64_t e = d + B;                                  // one past its last
  for (uint64_t i = a + threadIdx.x; i < b; i += static_cast<uint64_t>(BLOCK) * UNROLL) {
    uint4 lo[UNROLL], hi[UNROLL];
    uint32_t shift[UNROLL];
    bool interior[UNROLL];
    uint32_t rank[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint64_t k = i + static_cast<uint64_t>(u) * BLOCK;
      interior[u] = false;
      if (k < b) {
        const uint64_t x = (vbase + k) << 4;
        while (x >= e) {
          ++r;
          d = e;
          e += B;
        }
        rank[u] = r;
        if (x >= d && x + 16 <= e) {
          interior[u] = true;
          const uint64_t src = p.src[J.src0 + r] + (x - d);
          const uint32_t s = static_cast<uint32_t>(src & 15u);
          const uint4* blk = reinterpret_cast<const uint4*>(src - s);
          shift[u] = s;
          if (s == 0) {
            lo[u] = ld_nc_stream(blk);
            hi[u] = lo[u];
          } else {
            lo[u] = ld_nc_cached(blk);
            hi[u] = ld_nc_cached(blk + 1);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint64_t k = i + static_cast<uint64_t>(u) * BLOCK;
      if (k >= b) continue;
      const uint64_t x = (vbase + k) << 4;
      if (interior[u]) {
        st16(reinterpret_cast<uint4*>(x), realign16(lo[u], hi[u], shift[u]));
      } else {
        const uint32_t q0 = rank[u];
        const uint64_t dq = J.out + static_cast<uint64_t>(q0) * B;
        for (uint32_t j = 0; j < 16; ++j) {
          const uint64_t y = x + j;
          if (y < J.out || y >= out_end) continue;
          const bool next = y >= dq + B;  // byte of rank q0 + 1
          const uint8_t* src = reinterpret_cast<const uint8_t*>(p.src[J.src0 + q0 + (next ? 1 : 0)]);
          *reinterpret_cast<uint8_t*>(y) = src[y - dq - (next ? B : 0)];
        }
      }
    }
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
__global__ void __launch_bounds__(kGatherBlock, FLAT ? 4 : 2)
    dc_gather_kernel(const __grid_constant__ GatherParams<MAXJ, MAXS> p) {
  const uint64_t g0 = static_cast<uint64_t>(blockIdx.x) * p.chunk_vec;
  if (g0 >= p.total_vec) return;
  const uint64_t g1 = min(g0 + p.chunk_vec, p.total_vec);
  gather_cta<kGatherBlock, FLAT ? kGatherUnroll : kGatherUnrollGeneral, FLAT>(p, g0, g1);
}

// Single-CTA gather for small outputs: one CTA copies everything.
template <int MAXJ, int MAXS, bool FLAT>
__global__ void __launch_bounds__(FLAT ? kGatherSingleBlock : kGatherSingleBlockGeneral)
    dc_gather_single_kernel(const __grid_constant__ GatherParams<MAXJ, MAXS> p) {
  constexpr int kBlock = FLAT ? kGatherSingleBlock : kGatherSingleBlockGeneral;
  gather_cta<kBlock, FLAT ? kGatherUnroll : kGatherUnrollGeneral, FLAT>(p, 0, p.total_vec);
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
