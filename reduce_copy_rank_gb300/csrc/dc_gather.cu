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
//    gathers into one launch), numbered by a prefix over the jobs.  Vectors
//    are grouped in tiles of at most BLOCK x V; CTA c takes tiles c, c + G,
//    c + 2G, ... (G CTAs), so that all CTAs sweep the buffers together.  The
//    single-job kernels take their tile size from the launch, sized by the
//    planner so that every SM gets the same share of the output.
//  * Inside a tile, thread t takes vectors t, t + BLOCK, ..., across rank
//    boundaries: the flat loop of the page.  (The page's first version copied
//    rank by rank, leaving threads idle and serialising the ranks' reads.)  A
//    thread's vector index only grows, so it finds its rank (and job) by
//    walking forward: comparisons, one division when it enters a job, never
//    one per element.
//  * Aligned job (flat): 16-byte loads and stores, either held in registers
//    (mode 2) or staged through a per-thread cp.async ring in shared memory
//    (mode 3, the default: more bytes in flight without registers; a launch
//    in which every CTA has one tile loads straight into registers).
//  * Unaligned job: each output vector that lies inside one rank's bytes is
//    built from the two aligned source blocks that cover it with a funnel
//    shift, so loads and stores stay 16 bytes wide and aligned (registers,
//    mode 0; staged through a cp.async ring with per-rank affine state,
//    mode 5); the few vectors that straddle two ranks or stick out of the
//    output (at most P+1 per job) are assembled from each rank's part (one
//    or two aligned blocks) or from bytes, with their loads issued before
//    their stores; in mode 5 one extra CTA copies them beside the ring.
//  * all_gather_many (mode 4): the aligned jobs come first and are staged by
//    the first part of the grid, the unaligned ones by the rest; in these
//    parts each CTA takes a contiguous run of tiles, starting at a job the
//    host looked up, so that a thread enters only the jobs of its run.
//  * Jobs with fewer than kGatherSmallBytes per rank are assembled from bytes.
//  * Programmatic dependent launch: the single-job staged kernels prefetch
//    their first tile into L2 before they wait for the previous kernel of
//    the stream; the others trigger the next kernel and wait at entry.
#include <atomic>

#include "dc_device.cuh"
#include "dc_internal.h"

namespace dc {
namespace {

// Per-thread position among the jobs and ranks of a launch.  A thread's
// output vector indices only grow, so the cursor only moves forward: the job
// by comparison with the job table, the rank by comparison with the rank
// boundaries.  Entering a job costs one 64-bit division (the rank of the
// thread's first vector in it); after that, nothing per element but
// comparisons.
struct Cursor {
  int j;           // current job
  uint64_t jbeg;   // its first global vector
  uint64_t jend;   // one past its last
  bool fresh;      // rank state not yet set for job j
  uint32_t r;      // current rank
  uint64_t lo;     // flat: first job-local vector of rank r; unaligned: its first output byte
  uint64_t hi;     // one past its last (same units)
};

// Bounds checks of the checked build (in_bounds): a load of rank r of job J
// must lie in the 16-byte-block hull of that rank's source, a store in the
// job's output.  Sites, for the fault record: kSite* below.
enum : uint32_t {
  kSiteBytes = 100, kSiteFlat1 = 101, kSiteStaged1 = 102, kSiteStagedRing = 103, kSiteStagedJobs = 104,
  kSiteSpan = 105, kSiteBoundary = 106, kSiteRealign = 107, kSiteSmallVec = 108, kSiteRealignJobs = 109,
  kSiteSmallJobs = 110, kSiteGeneral = 111, kSitePrefetch = 112, kSiteWarpRealign = 113,
  kSiteWarpRealignJobs = 114,
};
template <int MAXJ, int MAXS>
__device__ __forceinline__ bool load_ok(const GatherParams<MAXJ, MAXS>& p, const GatherJob& J, uint32_t r,
                                        const void* a, uint64_t len, uint32_t site) {
  const uint64_t s = p.src[J.src0 + r];
  return in_bounds(a, len, hull_lo(s), hull_hi(s, J.bytes), site);
}
template <int MAXJ, int MAXS>
__device__ __forceinline__ bool store_ok(const GatherParams<MAXJ, MAXS>& p, const GatherJob& J, const void* a,
                                         uint64_t len, uint32_t site) {
  return in_bounds(a, len, J.out, J.out + static_cast<uint64_t>(p.P) * J.bytes, site);
}

template <int MAXJ, int MAXS>
__device__ __forceinline__ void cursor_to_job(const GatherParams<MAXJ, MAXS>& p, Cursor& c,
                                              uint64_t k) {
  while (k >= c.jend) {
    ++c.j;
    c.jbeg = p.job[c.j].vfirst;
    c.jend = c.jbeg + p.job[c.j].nvec;
    c.fresh = true;
  }
}

// The job holding global vector k (k < total_vec): the last job whose first
// vector is at or before k (jobs are numbered in vector order), found by
// binary search, so that a thread whose first vector lies deep in a long job
// table does not walk the table from its start.
template <int MAXJ, int MAXS>
__device__ __forceinline__ int job_of(const GatherParams<MAXJ, MAXS>& p, uint64_t k) {
  int lo = 0, hi = p.njobs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.job[mid].vfirst <= k)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// A cursor at the job holding global vector k (or at job 0 past the end).
template <int MAXJ, int MAXS>
__device__ __forceinline__ Cursor cursor_at(const GatherParams<MAXJ, MAXS>& p, uint64_t k) {
  const int j = k < p.total_vec ? job_of(p, k) : 0;
  return Cursor{j, p.job[j].vfirst, p.job[j].vfirst + p.job[j].nvec, true, 0, 0, 0};
}

// Flat job: rank r owns job-local vectors [r*vp, (r+1)*vp), vp = B/16.
template <int MAXJ, int MAXS>
__device__ __forceinline__ const uint4* flat_source(const GatherParams<MAXJ, MAXS>& p, Cursor& c,
                                                    const GatherJob& J, uint64_t kl) {
  const uint64_t vp = J.bytes >> 4;
  if (c.fresh) {
    c.r = static_cast<uint32_t>(kl / vp);
    c.lo = static_cast<uint64_t>(c.r) * vp;
    c.hi = c.lo + vp;
    c.fresh = false;
  }
  while (kl >= c.hi) {
    ++c.r;
    c.lo = c.hi;
    c.hi += vp;
  }
  return reinterpret_cast<const uint4*>(p.src[J.src0 + c.r]) + (kl - c.lo);
}

// Unaligned job: rank r owns output bytes [d_r, d_r + B), d_r = out + r*B;
// x is the first byte of the output vector.
template <int MAXJ, int MAXS>
__device__ __forceinline__ void unaligned_rank(Cursor& c, const GatherJob& J, uint64_t x) {
  if (c.fresh) {
    c.r = static_cast<uint32_t>((max(x, J.out) - J.out) / J.bytes);
    c.lo = J.out + static_cast<uint64_t>(c.r) * J.bytes;
    c.hi = c.lo + J.bytes;
    c.fresh = false;
  }
  while (x >= c.hi) {
    ++c.r;
    c.lo = c.hi;
    c.hi += J.bytes;
  }
}

// Bytes [x, x+16) of a job's output that are not one rank's aligned-source
// vector: copied one by one.  `r` is the rank of the vector's first output
// byte; for jobs of at least kGatherSmallBytes per rank the vector holds
// bytes of rank r and r+1 only, for smaller jobs the rank of each byte is
// found by a 32-bit division (the whole job is under kMaxRanks*128 bytes).
template <int MAXJ, int MAXS>
__device__ __forceinline__ void copy_bytes(const GatherParams<MAXJ, MAXS>& p, const GatherJob& J,
                                           uint64_t x, uint32_t r, bool small) {
  const uint64_t out_end = J.out + static_cast<uint64_t>(p.P) * J.bytes;
  for (uint32_t i = 0; i < 16; ++i) {
    const uint64_t y = x + i;
    if (y < J.out || y >= out_end) continue;
    uint32_t q;
    uint64_t off;
    if (small) {
      const uint32_t o = static_cast<uint32_t>(y - J.out), B = static_cast<uint32_t>(J.bytes);
      q = o / B;
      off = o - q * B;
    } else {
      const uint64_t d = J.out + static_cast<uint64_t>(r) * J.bytes;
      q = r + (y >= d + J.bytes ? 1u : 0u);
      off = y - d - (q > r ? J.bytes : 0);
    }
    const uint8_t* a = reinterpret_cast<const uint8_t*>(p.src[J.src0 + q]) + off;
    if (load_ok(p, J, q, a, 1, kSiteBytes) && store_ok(p, J, reinterpret_cast<void*>(y), 1, kSiteBytes))
      *reinterpret_cast<uint8_t*>(y) = *a;
  }
}

// Copy output vectors, tile by tile: tile t covers global vectors
// [t*TILE, (t+1)*TILE), TILE = BLOCK*UNROLL; this CTA takes tiles
// first, first + step, ...  Thread i of the CTA owns vectors
// t*TILE + i + u*BLOCK, u < UNROLL: all its loads are issued before its
// first store.
//  * Flat job vector: one LDG.128 from its rank's payload.
//  * Unaligned job vector lying inside one rank's bytes: source start s =
//    src address mod 16; the aligned block holding it and, if s != 0, the
//    next one; a funnel shift gives the 16 output bytes.  Both blocks hold
//    source bytes of this vector, so they lie in the source allocation.
//  * Any other vector (rank boundary, output ends, jobs under
//    kGatherSmallBytes per rank): byte copies.
// One aligned job (dc_all_gather with everything 16-byte aligned): the hot
// loop with the least state, so it fits the 32 registers of full occupancy.
// Idx is uint32_t when the output has fewer than 2^31 vectors (32 GiB).
template <int BLOCK, int UNROLL, typename Idx, int MAXS>
__device__ __forceinline__ void gather_tiles_flat1(const GatherParams<1, MAXS>& p, Idx first,
                                                   Idx step) {
  // the launch's tile (multi-CTA launches), else a full BLOCK*UNROLL
  const Idx tile = p.tile_vec > 0 && static_cast<Idx>(p.tile_vec) < static_cast<Idx>(BLOCK) * UNROLL
                       ? static_cast<Idx>(p.tile_vec)
                       : static_cast<Idx>(BLOCK) * UNROLL;
  const Idx total = static_cast<Idx>(p.total_vec);
  const Idx ntiles = (total + tile - 1) / tile;
  const Idx vp = static_cast<Idx>(p.job[0].bytes >> 4);
  uint4* out = reinterpret_cast<uint4*>(p.job[0].out);
  uint32_t r = 0;
  Idx rlo = 0, rhi = vp;
  bool fresh = true;
  for (Idx t = first; t < ntiles; t += step) {
    const Idx base = t * tile + threadIdx.x;
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const Idx k = base + static_cast<Idx>(u) * BLOCK;
      if (static_cast<Idx>(u) * BLOCK + threadIdx.x < tile && k < total) {
        if (fresh) {
          r = static_cast<uint32_t>(k / vp);
          rlo = static_cast<Idx>(r) * vp;
          rhi = rlo + vp;
          fresh = false;
        }
        while (k >= rhi) {
          ++r;
          rlo = rhi;
          rhi += vp;
        }
        const uint4* a = reinterpret_cast<const uint4*>(p.src[r]) + (k - rlo);
        if (load_ok(p, p.job[0], r, a, 16, kSiteFlat1)) v[u] = ld_nc_stream(a);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const Idx k = base + static_cast<Idx>(u) * BLOCK;
      if (static_cast<Idx>(u) * BLOCK + threadIdx.x < tile && k < total &&
          store_ok(p, p.job[0], out + k, 16, kSiteFlat1))
        st16(out + k, v[u]);
    }
  }
}

// One aligned job, staged through shared memory.  Same tiles and rank walk
// as gather_tiles_flat1 (tile = BLOCK*V vectors), but the loads are cp.async
// copies into a ring of S shared-memory slots per thread: while tile i is
// stored (shared -> registers -> STG.128), the copies of tiles i+1..i+S-1
// are already in flight, and in-flight data costs shared memory instead of
// registers (192 KB per SM instead of 128 KB).  Each thread only reads back
// the slots it filled itself, so no barrier is needed; the waits are
// cp.async.wait_group, a hardware wait on the thread's own copies.  When
// every CTA has one tile at most (outputs up to one full tile per resident
// CTA, 14.9 MB), there is nothing to overlap, and the loads go straight to
// registers: back to back, 8 x 128 KiB 2.02 -> 1.87 us per call, the same as
// the register kernel (mode 2).
template <int BLOCK, int V, int S, int MAXS>
__device__ __forceinline__ void gather_tiles_staged(const GatherParams<1, MAXS>& p, uint32_t first,
                                                    uint32_t step) {
  extern __shared__ uint4 stage_buf[];  // [S][V][BLOCK]
  const uint32_t tile = static_cast<uint32_t>(p.tile_vec);  // <= BLOCK*V
  const uint32_t total = static_cast<uint32_t>(p.total_vec);
  const uint32_t ntiles = (total + tile - 1) / tile;
  const uint32_t vp = static_cast<uint32_t>(p.job[0].bytes >> 4);
  uint4* out = reinterpret_cast<uint4*>(p.job[0].out);
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage_buf)) + 16u * threadIdx.x;
  uint32_t r = 0, rlo = 0, rhi = vp;
  bool fresh = true;
  if (ntiles <= step) {  // one tile per CTA: no ring, the loads go straight to registers
    uint4 v[V];
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint32_t i = u * BLOCK + threadIdx.x, k = first * tile + i;
      if (i < tile && k < total) {
        if (fresh) {
          r = k / vp;
          rlo = r * vp;
          rhi = rlo + vp;
          fresh = false;
        }
        while (k >= rhi) {
          ++r;
          rlo = rhi;
          rhi += vp;
        }
        const uint4* a = reinterpret_cast<const uint4*>(p.src[r]) + (k - rlo);
        if (load_ok(p, p.job[0], r, a, 16, kSiteStaged1)) v[u] = ld_nc_stream(a);
      }
    }
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint32_t i = u * BLOCK + threadIdx.x, k = first * tile + i;
      if (i < tile && k < total && store_ok(p, p.job[0], out + k, 16, kSiteStaged1)) st16(out + k, v[u]);
    }
    return;
  }
  auto issue = [&](uint32_t slot, uint32_t t) {
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint32_t i = u * BLOCK + threadIdx.x, k = t * tile + i;
      if (t < ntiles && i < tile && k < total) {
        if (fresh) {
          r = k / vp;
          rlo = r * vp;
          rhi = rlo + vp;
          fresh = false;
        }
        while (k >= rhi) {
          ++r;
          rlo = rhi;
          rhi += vp;
        }
        const uint4* a = reinterpret_cast<const uint4*>(p.src[r]) + (k - rlo);
        if (load_ok(p, p.job[0], r, a, 16, kSiteStagedRing)) cp_async16(sbase + 16u * BLOCK * (slot * V + u), a);
      }
    }
    cp_async_commit();  // one group per slot fill, empty past the last tile
  };
  uint32_t t_issue = first;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    issue(s, t_issue);
    t_issue += step;
  }
  uint32_t slot = 0;
  for (uint32_t t = first; t < ntiles; t += step) {
    cp_async_wait<S - 1>();  // the oldest group: tile t
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint32_t i = u * BLOCK + threadIdx.x, k = t * tile + i;
      if (i < tile && k < total && store_ok(p, p.job[0], out + k, 16, kSiteStagedRing))
        st16(out + k, ld_shared16(sbase + 16u * BLOCK * (slot * V + u)));
    }
    issue(slot, t_issue);  // refill the slot just drained
    t_issue += step;
    slot = (slot + 1 == S) ? 0 : slot + 1;
  }
  cp_async_wait<0>();
}

// The aligned jobs of a split launch (global vectors [0, flat_vec), jobs
// ordered aligned first), staged like gather_tiles_staged but over a job
// table: the issuing side walks jobs and ranks forward with a Cursor, the
// draining side walks jobs only (it needs each vector's output address).
// With many jobs (p.flat_per > 0), CTA `cta` of the part takes the
// contiguous run of flat_per tiles from tile cta * flat_per: a thread's
// vectors then lie close together and it enters only the few jobs of its
// run.  (With tiles dealt round robin, a thread's consecutive tiles are the
// whole part's share apart, so it crossed many jobs per tile, each a
// dependent read of the job table and a division: 250 aligned jobs of 4-64
// KiB x 4 ranks took 38 us.)  With few jobs (flat_per == 0) tiles are dealt
// round robin over the part's `nctas` CTAs, so that all CTAs sweep the
// buffers together (the six-tensor batch with 8 x 32 MiB in it: 2-3 %
// faster that way).  Either way the CTA starts at job p.flat_tab[cta],
// the job of its first vector (written by the host).
template <int BLOCK, int V, int S, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_tiles_staged_jobs(const GatherParams<MAXJ, MAXS>& p, uint32_t cta,
                                                         uint32_t nctas) {
  extern __shared__ uint4 stage_buf[];  // [S][V][BLOCK]
  constexpr uint64_t kTile = static_cast<uint64_t>(BLOCK) * V;
  const uint64_t total = p.flat_vec;
  const uint64_t ntiles = (total + kTile - 1) / kTile;
  const bool runs = p.flat_per != 0;
  const uint64_t t0 = runs ? static_cast<uint64_t>(cta) * p.flat_per : cta;
  const uint64_t t1 = runs ? min(t0 + p.flat_per, ntiles) : ntiles;
  const uint64_t ts = runs ? 1 : nctas;
  if (t0 >= t1) return;
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage_buf)) + 16u * threadIdx.x;
  const int j0 = MAXJ > 1 ? static_cast<int>(p.flat_tab[cta]) : 0;
  Cursor c{j0, p.job[j0].vfirst, p.job[j0].vfirst + p.job[j0].nvec, true, 0, 0, 0};
  int jd = c.j;
  uint64_t dbeg = c.jbeg, dend = c.jend;
  auto issue = [&](uint32_t slot, uint64_t t) {
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint64_t k = t * kTile + static_cast<uint64_t>(u) * BLOCK + threadIdx.x;
      if (t < t1 && k < total) {
        cursor_to_job(p, c, k);
        const uint4* a = flat_source(p, c, p.job[c.j], k - c.jbeg);
        if (load_ok(p, p.job[c.j], c.r, a, 16, kSiteStagedJobs)) cp_async16(sbase + 16u * BLOCK * (slot * V + u), a);
      }
    }
    cp_async_commit();
  };
  uint64_t t_issue = t0;
#pragma unroll
  for (int s = 0; s < S; ++s) {
    issue(s, t_issue);
    t_issue += ts;
  }
  uint32_t slot = 0;
  for (uint64_t t = t0; t < t1; t += ts) {
    cp_async_wait<S - 1>();
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint64_t k = t * kTile + static_cast<uint64_t>(u) * BLOCK + threadIdx.x;
      if (k < total) {
        while (k >= dend) {
          ++jd;
          dbeg = p.job[jd].vfirst;
          dend = dbeg + p.job[jd].nvec;
        }
        uint4* d = reinterpret_cast<uint4*>(p.job[jd].out) + (k - dbeg);
        if (store_ok(p, p.job[jd], d, 16, kSiteStagedJobs)) st16(d, ld_shared16(sbase + 16u * BLOCK * (slot * V + u)));
      }
    }
    issue(slot, t_issue);
    t_issue += ts;
    slot = (slot + 1 == S) ? 0 : slot + 1;
  }
  cp_async_wait<0>();
}

// The 16 source bytes starting at `a`, of which the first `len` (1..16) are
// wanted: the aligned blocks holding the first and the last wanted byte (the
// same block when the span does not cross a 16-byte boundary) funnel-shifted
// by a mod 16.  Both blocks hold wanted bytes, so both lie in the source
// allocation; bytes past `len` are whatever follows in those blocks.
// [hlo, hhi) is the source's block hull (for the checked build).
__device__ __forceinline__ uint4 load_span(const uint8_t* a, uint64_t len, uint64_t hlo, uint64_t hhi) {
  const uintptr_t ia = reinterpret_cast<uintptr_t>(a);
  const uint4* b0 = reinterpret_cast<const uint4*>(ia & ~static_cast<uintptr_t>(15));
  const uint4* b1 = reinterpret_cast<const uint4*>((ia + len - 1) & ~static_cast<uintptr_t>(15));
  uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
  if (in_bounds(b0, 16, hlo, hhi, kSiteSpan)) lo = ld_nc_stream(b0);
  if (in_bounds(b1, 16, hlo, hhi, kSiteSpan)) hi = ld_nc_stream(b1);
  return realign16_sel(lo, hi, static_cast<uint32_t>(ia & 15u));
}

// v's bytes moved up by n (0..15) places (byte i -> i + n; little-endian).
__device__ __forceinline__ void shift_up_bytes(uint64_t& lo, uint64_t& hi, uint32_t n) {
  if (n >= 8) {
    hi = lo << (8u * (n - 8u));
    lo = 0;
  } else if (n > 0) {
    hi = (hi << (8u * n)) | (lo >> (64u - 8u * n));
    lo <<= 8u * n;
  }
}

// A vector at a rank boundary of a job of at least kGatherSmallBytes per rank
// (x 16-byte aligned, r the rank of byte x; x may lie before the output or
// the vector stick out of its end).  Its output bytes [y0, y1) are the end of
// rank r's payload, [y0, z), and the start of rank r+1's, [z, y1): each part
// is one span of at most 16 source bytes, loaded as one or two aligned
// 16-byte blocks (all four loads issued together), shifted into place and
// merged; a vector inside the output is written with one 16-byte store, the
// first and last vector of the output byte by byte.
template <int MAXJ, int MAXS>
__device__ __forceinline__ void copy_boundary(const GatherParams<MAXJ, MAXS>& p, const GatherJob& J,
                                              uint64_t x, uint32_t r) {
  const uint64_t out_end = J.out + static_cast<uint64_t>(p.P) * J.bytes;
  const uint64_t d = J.out + static_cast<uint64_t>(r) * J.bytes;  // first output byte of rank r
  const uint64_t y0 = max(x, J.out), y1 = min(x + 16, out_end);
  const uint64_t z = min(d + J.bytes, y1);  // first output byte of rank r+1, or y1
  const uint8_t* s0 = reinterpret_cast<const uint8_t*>(p.src[J.src0 + r]);
  const uint8_t* s1 = r + 1 < static_cast<uint32_t>(p.P)
                          ? reinterpret_cast<const uint8_t*>(p.src[J.src0 + r + 1]) : s0;
  const uint64_t a0 = reinterpret_cast<uint64_t>(s0), a1 = reinterpret_cast<uint64_t>(s1);
  const uint4 va = load_span(s0 + (y0 - d), z - y0, hull_lo(a0), hull_hi(a0, J.bytes));
  const uint4 vb = z < y1 ? load_span(s1, y1 - z, hull_lo(a1), hull_hi(a1, J.bytes)) : va;
  uint64_t alo = va.x | (static_cast<uint64_t>(va.y) << 32), ahi = va.z | (static_cast<uint64_t>(va.w) << 32);
  uint64_t blo = vb.x | (static_cast<uint64_t>(vb.y) << 32), bhi = vb.z | (static_cast<uint64_t>(vb.w) << 32);
  const uint32_t na = static_cast<uint32_t>(y0 - x), nb = static_cast<uint32_t>(z - x);
  shift_up_bytes(alo, ahi, na);
  shift_up_bytes(blo, bhi, nb & 15u);
  // bytes [0, nb) from rank r, [nb, 16) from rank r+1
  const uint64_t mlo = nb >= 8 ? ~0ull : (1ull << (8u * nb)) - 1u;
  const uint64_t mhi = nb >= 16 ? ~0ull : nb <= 8 ? 0ull : (1ull << (8u * (nb - 8u))) - 1u;
  const uint64_t lo = (alo & mlo) | (blo & ~mlo), hi = (ahi & mhi) | (bhi & ~mhi);
  if (y0 == x && y1 == x + 16) {
    if (store_ok(p, J, reinterpret_cast<void*>(x), 16, kSiteBoundary))
      st16(reinterpret_cast<uint4*>(x), make_uint4(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32),
                                                    static_cast<uint32_t>(hi), static_cast<uint32_t>(hi >> 32)));
    return;
  }
  for (uint64_t y = y0; y < y1; ++y) {
    const uint32_t i = static_cast<uint32_t>(y - x);
    if (store_ok(p, J, reinterpret_cast<void*>(y), 1, kSiteBoundary))
      *reinterpret_cast<uint8_t*>(y) =
          static_cast<uint8_t>((i < 8 ? lo >> (8u * i) : hi >> (8u * (i - 8u))) & 0xFFu);
  }
}

// Forward walk over the ranks of one unaligned job, in output-vector units.
// Output vector k is x(k) = xbase + 16k, xbase = out rounded down to 16.
// Rank r owns output bytes [d, d + B), d = out + r*B; the vectors wholly
// inside it are k in [klo, khi), klo = ceil((d - xbase)/16), khi =
// floor((d + B - xbase)/16).  For those the source start is src_r + x(k) -
// d, whose offset in its 16-byte block, s = (src_r + xbase - d) mod 16, is
// the same for every k, and whose block is base + k with base = (src_r +
// xbase - d - s) / 16: all of it computed once per rank.  The vectors in
// between (k < klo, or k >= khi in the last rank) straddle two ranks or an
// end of the output.
template <typename Idx>
struct RankWalk {
  uint32_t r;
  uint32_t s;
  Idx klo, khi;
  uint64_t base;  // block address of vector k: base + 16k, formed only for k in [klo, khi)
  bool fresh;
};

template <typename Idx, int MAXJ, int MAXS>
__device__ __forceinline__ void rank_enter(RankWalk<Idx>& w, const GatherParams<MAXJ, MAXS>& p,
                                           const GatherJob& J, uint64_t xbase) {
  const uint64_t d = J.out + static_cast<uint64_t>(w.r) * J.bytes;
  w.klo = static_cast<Idx>((d - xbase + 15) >> 4);
  w.khi = static_cast<Idx>((d + J.bytes - xbase) >> 4);
  const uint64_t a = p.src[J.src0 + w.r] + xbase - d;  // source address that x(0) would map to
  w.s = static_cast<uint32_t>(a & 15u);
  w.base = a - w.s;  // modulo 2^64: it may lie outside every allocation
}

// Idx is uint32_t when the whole output (from out rounded down to 16) is
// under 4 GiB, so that 16k and every rank size fit 32 bits.
template <typename Idx, int MAXJ, int MAXS>
__device__ __forceinline__ void walk_to(RankWalk<Idx>& w, const GatherParams<MAXJ, MAXS>& p,
                                        const GatherJob& J, uint64_t xbase, Idx k) {
  if (w.fresh) {
    const Idx lead = static_cast<Idx>(J.out - xbase);  // output bytes before out in vector 0
    const Idx x = static_cast<Idx>(16) * k;            // relative to xbase
    w.r = static_cast<uint32_t>((x > lead ? x - lead : Idx(0)) / static_cast<Idx>(J.bytes));
    rank_enter(w, p, J, xbase);
    w.fresh = false;
  }
  while (k >= w.khi && w.r + 1 < static_cast<uint32_t>(p.P)) {
    ++w.r;
    rank_enter(w, p, J, xbase);
  }
}

// One unaligned job (at least kGatherSmallBytes per rank), staged through
// shared memory.  Issuing side (rank walk above): vector k inside rank r
// copies block base + k and, if s != 0, the next one (both hold source bytes
// of the vector, so both lie in the source allocation) with cp.async into
// the thread's ring slot, and notes s and "inside one rank" in 5 bits of a
// register (S*V*5 <= 32 bits).  Draining side: the funnel shift of the two
// blocks by s gives the 16 output bytes, one 16-byte store.  No barrier:
// each thread reads back only the slots it filled.  The vectors that are not
// inside one rank (the ones holding d_b = out + b*B, b in [0, P], with d_b
// not 16-byte aligned; B >= 16) are skipped here: the launch's last CTA
// copies them (copy_boundaries), so their memory round trip runs beside the
// ring instead of after a ring thread's last tile.
template <int BLOCK, int V, int S, typename Idx, int MAXS>
__device__ __forceinline__ void gather_tiles_staged_realign(const GatherParams<1, MAXS>& p,
                                                            Idx first, Idx step) {
  static_assert(S * V * 5 <= 32, "ring notes must fit one register");
  extern __shared__ uint4 stage_buf[];  // [S][V][2][BLOCK]
  const GatherJob& J = p.job[0];
  // <= BLOCK*V; outputs of 4 GiB or more (64-bit indices) always take full
  // tiles, which keeps that instance of the loop within its registers
  const Idx tile = sizeof(Idx) == 4 ? static_cast<Idx>(p.tile_vec) : static_cast<Idx>(BLOCK) * V;
  const Idx total = static_cast<Idx>(p.total_vec);
  const Idx ntiles = (total + tile - 1) / tile;
  // this thread's vectors of a tile: u*BLOCK + threadIdx.x < tile for u < nv
  const int nv = threadIdx.x < tile ? static_cast<int>((tile - threadIdx.x + BLOCK - 1) / BLOCK) : 0;
  const uint64_t xbase = J.out & ~static_cast<uint64_t>(15);
  uint4* const out = reinterpret_cast<uint4*>(xbase);
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage_buf)) + 16u * threadIdx.x;
  RankWalk<Idx> w{0, 0, 0, 0, 0, true};
  uint32_t notes = 0;  // 5 bits per ring vector: s | inside << 4
  auto slot_addr = [&](uint32_t slot, int u, int h) {
    return sbase + 16u * BLOCK * static_cast<uint32_t>((slot * V + u) * 2 + h);
  };
  auto issue = [&](uint32_t slot, Idx t) {
    notes &= ~(((1u << (5 * V)) - 1u) << (5 * V * slot));
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const Idx k = t * tile + static_cast<Idx>(u) * BLOCK + threadIdx.x;
      if (t < ntiles && u < nv && k < total) {
        walk_to(w, p, J, xbase, k);
        if (k >= w.klo && k < w.khi) {
          const uint4* blk = reinterpret_cast<const uint4*>(w.base + 16 * static_cast<uint64_t>(k));
          if (load_ok(p, J, w.r, blk, 16, kSiteRealign))
            cp_async16_ca(slot_addr(slot, u, 0), blk);  // block k+1 of a thread is
          if (w.s && load_ok(p, J, w.r, blk + 1, 16, kSiteRealign))
            cp_async16_ca(slot_addr(slot, u, 1), blk + 1);  // block k of its neighbour
          notes |= (w.s | 16u) << (5 * (slot * V + u));
        }
      }
    }
    cp_async_commit();
  };
  Idx t_issue = first;
#pragma unroll
  for (int i = 0; i < S; ++i) {
    issue(i, t_issue);
    t_issue += step;
  }
  uint32_t slot = 0;
  for (Idx t = first; t < ntiles; t += step) {
    cp_async_wait<S - 1>();
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const Idx k = t * tile + static_cast<Idx>(u) * BLOCK + threadIdx.x;
      if (u < nv && k < total) {
        const uint32_t m = (notes >> (5 * (slot * V + u))) & 31u;
        if (m & 16u) {  // inside one rank (the others: copy_boundaries)
          const uint32_t sh = m & 15u;
          const uint4 lo = ld_shared16(slot_addr(slot, u, 0));
          const uint4 hi = sh ? ld_shared16(slot_addr(slot, u, 1)) : lo;
          if (store_ok(p, J, out + k, 16, kSiteRealign)) st16(out + k, realign16_sel(lo, hi, sh));
        }
      }
    }
    issue(slot, t_issue);
    t_issue += step;
    slot = (slot + 1 == S) ? 0 : slot + 1;
  }
  cp_async_wait<0>();
}

// One unaligned job (at least kGatherSmallBytes per rank, 32-bit indices),
// realigned across the lanes of a warp: the register path with far fewer
// instructions per vector than the shared-memory ring of
// gather_tiles_staged_realign, which ncu showed issue-bound (8 x (1 MiB+1 B):
// 3.9 M warp instructions against 1.2 M for the aligned copy, issue slots 66 %
// busy, almost no memory stalls).  Tiles as there; thread i of a tile takes
// vectors i, i + BLOCK, ... (V of them), so the 32 lanes of a warp hold 32
// consecutive output vectors.  A vector k inside rank r (k in [klo, khi), see
// RankWalk) is bytes [16k + s, 16k + s + 16) of the 16-byte blocks base_r +
// 16k and base_r + 16(k+1): each lane loads only the first block, straight
// into registers, and takes the second from the next lane (__shfl_down_sync),
// which loaded it as its own first block -- unless the next lane's vector is
// not vector k + 1 of the same rank (lane 31, the tile's last vector, the
// rank's last whole vector), in which case the lane loads its second block
// itself, in the same round of loads.  All loads of a thread's V vectors are
// issued before the first shuffle and store.  The vectors that are not inside
// one rank are left to the launch's last CTA (copy_boundaries), as in mode 5.
template <int BLOCK, int V, int MAXS>
__device__ __forceinline__ void gather_tiles_warp_realign(const GatherParams<1, MAXS>& p, uint32_t first,
                                                          uint32_t step) {
  const GatherJob& J = p.job[0];
  const uint32_t tile = static_cast<uint32_t>(p.tile_vec);  // <= BLOCK*V
  const uint32_t total = static_cast<uint32_t>(p.total_vec);
  const uint32_t ntiles = (total + tile - 1) / tile;
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t xbase = J.out & ~static_cast<uint64_t>(15);
  uint4* const out = reinterpret_cast<uint4*>(xbase);
  RankWalk<uint32_t> w{0, 0, 0, 0, 0, true};
  for (uint32_t t = first; t < ntiles; t += step) {
    uint4 lo[V], hi[V];
    uint32_t meta[V];  // s | inside << 4 | own second block << 5
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint32_t i = u * BLOCK + threadIdx.x, k = t * tile + i;
      meta[u] = 0;
      if (i < tile && k < total) {
        walk_to(w, p, J, xbase, k);
        if (k >= w.klo && k < w.khi) {
          const bool own_hi = w.s != 0 && (lane == 31u || k + 1 >= w.khi || i + 1 >= tile);
          const uint4* blk = reinterpret_cast<const uint4*>(w.base + 16 * static_cast<uint64_t>(k));
          if (load_ok(p, J, w.r, blk, 16, kSiteWarpRealign)) lo[u] = ld_nc_cached(blk);
          if (own_hi && load_ok(p, J, w.r, blk + 1, 16, kSiteWarpRealign)) hi[u] = ld_nc_cached(blk + 1);
          meta[u] = w.s | 16u | (own_hi ? 32u : 0u);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < V; ++u) {
      // every lane takes part in the shuffles; a lane whose next lane holds
      // vector k + 1 of the same rank uses that lane's first block
      uint4 nb;
      nb.x = __shfl_down_sync(0xffffffffu, lo[u].x, 1);
      nb.y = __shfl_down_sync(0xffffffffu, lo[u].y, 1);
      nb.z = __shfl_down_sync(0xffffffffu, lo[u].z, 1);
      nb.w = __shfl_down_sync(0xffffffffu, lo[u].w, 1);
      const uint32_t m = meta[u];
      if (m & 16u) {
        const uint32_t sh = m & 15u;
        const uint4 second = (m & 32u) ? hi[u] : nb;
        const uint32_t k = t * tile + u * BLOCK + threadIdx.x;
        if (store_ok(p, J, out + k, 16, kSiteWarpRealign)) st16(out + k, sh ? realign16_sel(lo[u], second, sh) : lo[u]);
      }
    }
  }
}

// The rank-boundary vectors of one unaligned job (at least
// kGatherSmallBytes per rank): thread b copies the vector holding d_b = out +
// b*B, b in [0, P], if d_b is not 16-byte aligned (the byte before d_b is
// rank b-1's, or lies before the output for b = 0).
template <int BLOCK, int MAXS>
__device__ __forceinline__ void copy_boundaries(const GatherParams<1, MAXS>& p) {
  const GatherJob& J = p.job[0];
  for (uint32_t b = threadIdx.x; b <= static_cast<uint32_t>(p.P); b += BLOCK) {
    const uint64_t d = J.out + static_cast<uint64_t>(b) * J.bytes;
    if (d & 15u) copy_boundary(p, J, d & ~static_cast<uint64_t>(15), b == 0 ? 0u : b - 1);
  }
}

// Bytes [x, x+16) of a job of fewer than kGatherSmallBytes per rank (the
// whole job is under kMaxRanks*128 bytes, so 32-bit offsets): the rank of
// the first byte by one division, then byte by byte forward; all 16 loads
// are issued before the first store.
template <int MAXJ, int MAXS>
__device__ __forceinline__ void copy_small_vector(const GatherParams<MAXJ, MAXS>& p, const GatherJob& J,
                                                  uint64_t x) {
  const uint64_t out_end = J.out + static_cast<uint64_t>(p.P) * J.bytes;
  const uint32_t B = static_cast<uint32_t>(J.bytes);
  const uint32_t lead = x < J.out ? static_cast<uint32_t>(J.out - x) : 0u;  // bytes before the output
  const uint32_t o0 = static_cast<uint32_t>(x + lead - J.out);
  uint32_t q = o0 / B, off = o0 - q * B;
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (uint32_t i = 0; i < 16; ++i) {
    if (i >= lead && x + i < out_end) {
      const uint8_t* a = reinterpret_cast<const uint8_t*>(p.src[J.src0 + q]) + off;
      const uint32_t b = load_ok(p, J, q, a, 1, kSiteSmallVec) ? __ldg(a) : 0u;
      w[i >> 2] |= b << (8u * (i & 3u));
      if (++off == B) {
        ++q;
        off = 0;
      }
    }
  }
  if (lead == 0 && x + 16 <= out_end) {
    if (store_ok(p, J, reinterpret_cast<void*>(x), 16, kSiteSmallVec))
      st16(reinterpret_cast<uint4*>(x), make_uint4(w[0], w[1], w[2], w[3]));
    return;
  }
#pragma unroll
  for (uint32_t i = 0; i < 16; ++i)
    if (i >= lead && x + i < out_end && store_ok(p, J, reinterpret_cast<void*>(x + i), 1, kSiteSmallVec))
      *reinterpret_cast<uint8_t*>(x + i) = static_cast<uint8_t>(w[i >> 2] >> (8u * (i & 3u)));
}

// The unaligned jobs of a split launch (global vectors [voff, vend), after
// the aligned jobs), through the same kind of shared-memory ring as
// gather_tiles_staged_realign.  The issuing side walks jobs forward and,
// inside a job of at least kGatherSmallBytes per rank, its ranks (RankWalk
// in job-local vector units); the draining side walks jobs only, for each
// vector's output address, and reads the vector's shift and kind from the
// register notes.  A vector of a smaller job (copy_small_vector) or at a
// rank boundary or output end (copy_boundary) is copied with its loads
// issued before its stores, so it costs one memory round trip.
template <int BLOCK, int V, int S, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_tiles_staged_realign_jobs(const GatherParams<MAXJ, MAXS>& p,
                                                                 uint32_t cta, uint32_t nctas, uint64_t voff,
                                                                 uint64_t vend) {
  static_assert(S * V * 5 <= 32, "ring notes must fit one register");
  extern __shared__ uint4 stage_buf[];  // [S][V][2][BLOCK]
  constexpr uint64_t kTile = static_cast<uint64_t>(BLOCK) * V;
  const uint64_t total = vend;
  const uint64_t ntiles = (total - voff + kTile - 1) / kTile;
  // CTA `cta` of the part: with many jobs (p.real_per > 0) the contiguous
  // run of real_per tiles from tile cta * real_per, with few jobs tiles cta,
  // cta + nctas, ... (as gather_tiles_staged_jobs); either way starting at
  // job p.real_tab[cta], the job of its first vector, written by the host
  // (a binary search here spilled registers, and walking the table from its
  // start cost a dependent read per job: 250 jobs of 128 B-4 KiB x 4 ranks
  // at +1 B took 36 us)
  const bool runs = p.real_per != 0;
  const uint64_t t0 = runs ? static_cast<uint64_t>(cta) * p.real_per : cta;
  const uint64_t t1 = runs ? min(t0 + p.real_per, ntiles) : ntiles;
  const uint64_t ts = runs ? 1 : nctas;
  if (t0 >= t1) return;
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(stage_buf)) + 16u * threadIdx.x;
  // issuing side: job j (vectors [jbeg, jend)), its ranks
  int j = MAXJ > 1 ? static_cast<int>(p.real_tab[cta]) : 0;
  uint64_t jbeg = p.job[j].vfirst, jend = jbeg + p.job[j].nvec;
  RankWalk<uint64_t> w{0, 0, 0, 0, 0, true};
  // draining side: job jd (vectors [dbeg, dend))
  int jd = j;
  uint64_t dbeg = jbeg, dend = jend;
  uint32_t notes = 0;  // 5 bits per ring vector: s | inside << 4
  auto slot_addr = [&](uint32_t slot, int u, int h) {
    return sbase + 16u * BLOCK * static_cast<uint32_t>((slot * V + u) * 2 + h);
  };
  auto issue = [&](uint32_t slot, uint64_t t) {
    notes &= ~(((1u << (5 * V)) - 1u) << (5 * V * slot));
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint64_t k = voff + t * kTile + static_cast<uint64_t>(u) * BLOCK + threadIdx.x;
      if (t < t1 && k < total) {
        while (k >= jend) {
          ++j;
          jbeg = p.job[j].vfirst;
          jend = jbeg + p.job[j].nvec;
          w.fresh = true;
        }
        const GatherJob& J = p.job[j];
        if (!(J.flags & kJobSmall)) {
          const uint64_t xbase = J.out & ~static_cast<uint64_t>(15);
          const uint64_t kl = k - jbeg;
          walk_to(w, p, J, xbase, kl);
          if (kl >= w.klo && kl < w.khi) {
            const uint4* blk = reinterpret_cast<const uint4*>(w.base + 16 * kl);
            if (load_ok(p, J, w.r, blk, 16, kSiteRealignJobs)) cp_async16_ca(slot_addr(slot, u, 0), blk);
            if (w.s && load_ok(p, J, w.r, blk + 1, 16, kSiteRealignJobs))
              cp_async16_ca(slot_addr(slot, u, 1), blk + 1);
            notes |= (w.s | 16u) << (5 * (slot * V + u));
          }
        }
      }
    }
    cp_async_commit();
  };
  uint64_t t_issue = t0;
#pragma unroll
  for (int i = 0; i < S; ++i) {
    issue(i, t_issue);
    t_issue += ts;
  }
  uint32_t slot = 0;
  for (uint64_t t = t0; t < t1; t += ts) {
    cp_async_wait<S - 1>();
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint64_t k = voff + t * kTile + static_cast<uint64_t>(u) * BLOCK + threadIdx.x;
      if (k < total) {
        while (k >= dend) {
          ++jd;
          dbeg = p.job[jd].vfirst;
          dend = dbeg + p.job[jd].nvec;
        }
        const GatherJob& J = p.job[jd];
        const uint64_t xbase = J.out & ~static_cast<uint64_t>(15);
        const uint64_t kl = k - dbeg;
        const uint32_t m = (notes >> (5 * (slot * V + u))) & 31u;
        if (m & 16u) {
          const uint32_t sh = m & 15u;
          const uint4 lo = ld_shared16(slot_addr(slot, u, 0));
          const uint4 hi = sh ? ld_shared16(slot_addr(slot, u, 1)) : lo;
          uint4* d = reinterpret_cast<uint4*>(xbase) + kl;
          if (store_ok(p, J, d, 16, kSiteRealignJobs)) st16(d, realign16_sel(lo, hi, sh));
        } else {
          const uint64_t x = xbase + 16 * kl;
          if (J.flags & kJobSmall)
            copy_small_vector(p, J, x);
          else
            copy_boundary(p, J, x, x < J.out ? 0u : static_cast<uint32_t>((x - J.out) / J.bytes));
        }
      }
    }
    issue(slot, t_issue);
    t_issue += ts;
    slot = (slot + 1 == S) ? 0 : slot + 1;
  }
  cp_async_wait<0>();
}

// The unaligned jobs of a split launch (global vectors [voff, vend)),
// realigned across the lanes of a warp in registers, as
// gather_tiles_warp_realign does for one job: lane i of a warp loads the
// first source block of its vector k and takes the second one from lane
// i + 1, which holds vector k + 1; a lane whose neighbour is in another rank
// or job, lane 31, and the last vector of a tile load their own second block.
// Tiles are dealt as in gather_tiles_staged_realign_jobs (runs for many
// jobs, round robin for few, from the job p.real_tab[cta]); a thread walks
// jobs and ranks forward.  The vectors not inside one rank (at most P+1 per
// job) are skipped here and copied by the part's boundary CTAs
// (copy_boundaries_jobs), beside the tiles: copied inline, their byte
// assembly spilled this part's registers.
template <int BLOCK, int V, typename Idx, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_tiles_warp_realign_jobs(const GatherParams<MAXJ, MAXS>& p, uint32_t cta,
                                                               uint32_t nctas, Idx voff, Idx vend) {
  constexpr Idx kTile = static_cast<Idx>(BLOCK) * V;
  const Idx ntiles = (vend - voff + kTile - 1) / kTile;
  const bool runs = p.real_per != 0;
  const Idx t0 = runs ? static_cast<Idx>(cta) * static_cast<Idx>(p.real_per) : static_cast<Idx>(cta);
  const Idx t1 = runs ? min(t0 + static_cast<Idx>(p.real_per), ntiles) : ntiles;
  const Idx ts = runs ? 1 : static_cast<Idx>(nctas);
  const uint32_t lane = threadIdx.x & 31u;
  int j = MAXJ > 1 ? static_cast<int>(p.real_tab[cta]) : 0;
  Idx jbeg = static_cast<Idx>(p.job[j].vfirst), jend = jbeg + static_cast<Idx>(p.job[j].nvec);
  RankWalk<Idx> w{0, 0, 0, 0, 0, true};
  for (Idx t = t0; t < t1; t += ts) {
    uint4 lo[V], hi[V];
    uint64_t dst[V];
    uint32_t meta[V];  // s | inside << 4 | own second block << 5 | store in bounds << 6
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const Idx i = static_cast<Idx>(u) * BLOCK + threadIdx.x;
      const Idx k = voff + t * kTile + i;
      meta[u] = 0;
      if (k < vend) {
        while (k >= jend) {
          ++j;
          jbeg = static_cast<Idx>(p.job[j].vfirst);
          jend = jbeg + static_cast<Idx>(p.job[j].nvec);
          w.fresh = true;
        }
        const GatherJob& J = p.job[j];
        const uint64_t xbase = J.out & ~static_cast<uint64_t>(15);
        const Idx kl = k - jbeg;
        walk_to(w, p, J, xbase, kl);
        dst[u] = xbase + 16 * static_cast<uint64_t>(kl);
        if (kl >= w.klo && kl < w.khi) {
          const bool own_hi = w.s != 0 && (lane == 31u || kl + 1 >= w.khi || i + 1 >= kTile);
          const uint4* blk = reinterpret_cast<const uint4*>(w.base + 16 * static_cast<uint64_t>(kl));
          if (load_ok(p, J, w.r, blk, 16, kSiteWarpRealignJobs)) lo[u] = ld_nc_cached(blk);
          if (own_hi && load_ok(p, J, w.r, blk + 1, 16, kSiteWarpRealignJobs)) hi[u] = ld_nc_cached(blk + 1);
          // (the checked build tests the store against this vector's job
          // here: by the store, the thread may have entered the next job)
          const bool sok = store_ok(p, J, reinterpret_cast<void*>(dst[u]), 16, kSiteWarpRealignJobs);
          meta[u] = w.s | 16u | (own_hi ? 32u : 0u) | (sok ? 64u : 0u);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < V; ++u) {
      uint4 nb;  // every lane takes part in the shuffles
      nb.x = __shfl_down_sync(0xffffffffu, lo[u].x, 1);
      nb.y = __shfl_down_sync(0xffffffffu, lo[u].y, 1);
      nb.z = __shfl_down_sync(0xffffffffu, lo[u].z, 1);
      nb.w = __shfl_down_sync(0xffffffffu, lo[u].w, 1);
      const uint32_t m = meta[u];
      if (m & 16u) {
        const uint32_t sh = m & 15u;
        const uint4 second = (m & 32u) ? hi[u] : nb;
        if (m & 64u) st16(reinterpret_cast<uint4*>(dst[u]), sh ? realign16_sel(lo[u], second, sh) : lo[u]);
      }
    }
  }
}

// The rank-boundary vectors of the unaligned jobs of a split launch (jobs
// [p.real_tab[0], p.small_job0)), copied by `nctas` CTAs: pair (job j, b),
// b in [0, P], is the vector holding d_b = out_j + b*B_j if d_b is not
// 16-byte aligned (as copy_boundaries does for one job).
template <int BLOCK, int MAXJ, int MAXS>
__device__ __forceinline__ void copy_boundaries_jobs(const GatherParams<MAXJ, MAXS>& p, uint32_t cta,
                                                     uint32_t nctas) {
  const uint32_t j0 = MAXJ > 1 ? p.real_tab[0] : 0;
  const uint32_t P1 = static_cast<uint32_t>(p.P) + 1;
  const uint32_t pairs = (static_cast<uint32_t>(p.small_job0) - j0) * P1;
  for (uint32_t idx = cta * BLOCK + threadIdx.x; idx < pairs; idx += nctas * BLOCK) {
    const uint32_t jj = idx / P1, b = idx - jj * P1;
    const GatherJob& J = p.job[j0 + jj];
    const uint64_t d = J.out + static_cast<uint64_t>(b) * J.bytes;
    if (d & 15u) copy_boundary(p, J, d & ~static_cast<uint64_t>(15), b == 0 ? 0u : b - 1);
  }
}

// The jobs of fewer than kGatherSmallBytes bytes per rank of a split launch
// (jobs [small_job0, njobs), global vectors [small_vec, total_vec)), copied by
// the launch's last `nctas` CTAs.  CTA c takes the contiguous run of
// small_per vectors starting small_per * c after small_vec; the host wrote in
// small_tab[c] and small_tab[c + 1] the jobs of its first and last vector.
// The CTA first copies those jobs' entries and source pointers from the
// parameter block into shared memory -- only those: parameters read at
// lane-dependent addresses are served one address at a time, and after an L2
// flush each new line is a miss, so copying the whole table of a large batch
// cost 138 us per call (120 tensors x 8 ranks) against 5 us warm -- so that
// the per-byte source reads of lanes in different jobs or ranks become
// shared-memory loads.  Then SPLIT threads share each 16-byte output vector
// (thread i takes bytes [(i % SPLIT) * 16/SPLIT, ...) of the CTA's vector i /
// SPLIT), find the vector's job by binary search in the shared table and
// assemble their bytes, all loads issued before the store.  Measured on GB300
// (120 tensors of 3..100 B x 8 ranks at +1 B, 20 calls back to back): 23 us
// per call before this part existed; 6.1, 5.1 and 5.15 us with 1, 2 and 4
// threads per vector (4 spreads the part over 4x the SMs and was best for 250
// tensors of 1..40 B x 4 ranks, 6.5 us, and for 16 tensors x 64 ranks, 3.9
// us); reading the parameters at warp-uniform addresses instead (one
// broadcast per word, 32 words per lane round) was 0.9-1.3 us slower.
template <int BLOCK, int SPLIT, int MAXJ, int MAXS>
__device__ __forceinline__ void copy_small_jobs(const GatherParams<MAXJ, MAXS>& p, uint32_t cta) {
  static_assert(SPLIT == 1 || SPLIT == 2 || SPLIT == 4, "16 bytes per vector");
  static_assert(MAXJ > 1, "split launches only");
  constexpr uint32_t kBytes = 16 / SPLIT;
  extern __shared__ uint4 stage_buf[];
  if (cta >= static_cast<uint32_t>(kMaxSmallCtas)) return;
  const int jlo = p.small_job0 + p.small_tab[cta], jhi = p.small_job0 + p.small_tab[cta + 1];
  if (jlo > jhi || jhi >= p.njobs) return;
  const int nj = jhi - jlo + 1;
  const uint32_t P = static_cast<uint32_t>(p.P);
  GatherJob* sj = reinterpret_cast<GatherJob*>(stage_buf);
  uint64_t* ssrc = reinterpret_cast<uint64_t*>(sj + nj);
  const uint32_t s0 = p.job[jlo].src0, ns = static_cast<uint32_t>(nj) * P;
  for (int i = threadIdx.x; i < nj; i += BLOCK) sj[i] = p.job[jlo + i];
  for (uint32_t i = threadIdx.x; i < ns; i += BLOCK) ssrc[i] = p.src[s0 + i];
  __syncthreads();
  const uint64_t k0 = p.small_vec + static_cast<uint64_t>(cta) * p.small_per;
  const uint64_t k1 = min(k0 + p.small_per, p.total_vec);
  for (uint64_t g = threadIdx.x; k0 + g / SPLIT < k1; g += BLOCK) {
    const uint64_t k = k0 + g / SPLIT;
    const uint32_t part = static_cast<uint32_t>(g % SPLIT) * kBytes;
    int lo = 0, hi = nj - 1;  // the last job whose first vector is at or before k
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sj[mid].vfirst <= k)
        lo = mid;
      else
        hi = mid - 1;
    }
    const uint64_t out = sj[lo].out, vfirst = sj[lo].vfirst;
    const uint32_t B = static_cast<uint32_t>(sj[lo].bytes), src0 = sj[lo].src0 - s0;
    const uint64_t x = (((out >> 4) + (k - vfirst)) << 4) + part;  // this thread's first byte
    const uint64_t out_end = out + static_cast<uint64_t>(P) * B;
    if (x >= out_end) continue;
    const uint32_t lead = x < out ? static_cast<uint32_t>(min(out - x, static_cast<uint64_t>(kBytes))) : 0u;
    const uint32_t o0 = static_cast<uint32_t>(x + lead - out);
    uint32_t q = o0 / B, off = o0 - q * B;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (uint32_t i = 0; i < kBytes; ++i) {
      if (i >= lead && x + i < out_end) {
        const uint64_t sa = ssrc[src0 + q];
        const uint8_t* a = reinterpret_cast<const uint8_t*>(sa) + off;
        const uint32_t b = in_bounds(a, 1, hull_lo(sa), hull_hi(sa, B), kSiteSmallJobs) ? __ldg(a) : 0u;
        w[i >> 2] |= b << (8u * (i & 3u));
        if (++off == B) {
          ++q;
          off = 0;
        }
      }
    }
    if (lead == 0 && x + kBytes <= out_end) {
      if (!in_bounds(reinterpret_cast<void*>(x), kBytes, out, out_end, kSiteSmallJobs)) continue;
      if constexpr (kBytes == 16)
        st16(reinterpret_cast<uint4*>(x), make_uint4(w[0], w[1], w[2], w[3]));
      else if constexpr (kBytes == 8)
        *reinterpret_cast<uint2*>(x) = make_uint2(w[0], w[1]);
      else
        *reinterpret_cast<uint32_t*>(x) = w[0];
    } else {
#pragma unroll
      for (uint32_t i = 0; i < kBytes; ++i)
        if (i >= lead && x + i < out_end &&
            in_bounds(reinterpret_cast<void*>(x + i), 1, out, out_end, kSiteSmallJobs))
          *reinterpret_cast<uint8_t*>(x + i) = static_cast<uint8_t>(w[i >> 2] >> (8u * (i & 3u)));
    }
  }
}

// voff: the tiles cover global vectors [voff, total_vec) (a split launch
// gives the vectors below voff to other CTAs).
template <int BLOCK, int UNROLL, bool FLAT, bool FAST_EDGES, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_tiles(const GatherParams<MAXJ, MAXS>& p, uint64_t first,
                                             uint64_t step, uint64_t voff = 0) {
  constexpr uint64_t kTile = static_cast<uint64_t>(BLOCK) * UNROLL;
  const uint64_t ntiles = (p.total_vec - voff + kTile - 1) / kTile;
  Cursor c = cursor_at(p, voff + first * kTile + threadIdx.x);
  for (uint64_t t = first; t < ntiles; t += step) {
    const uint64_t base = voff + t * kTile + threadIdx.x;
    uint4 lo[UNROLL], hi[UNROLL];
    uint64_t dst[UNROLL];
    uint32_t meta[UNROLL];  // FLAT: unused; else shift | kind << 8 | rank << 16
    int job[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint64_t k = base + static_cast<uint64_t>(u) * BLOCK;
      dst[u] = 0;
      if (k >= p.total_vec) continue;
      cursor_to_job(p, c, k);
      const GatherJob& J = p.job[c.j];
      const uint64_t kl = k - c.jbeg;
      job[u] = c.j;
      if (FLAT) {
        const uint4* a = flat_source(p, c, J, kl);
        if (load_ok(p, J, c.r, a, 16, kSiteGeneral)) lo[u] = ld_nc_stream(a);
        dst[u] = J.out + 16 * kl;
        continue;
      }
      if (J.flags & kJobFlat) {
        const uint4* a = flat_source(p, c, J, kl);
        if (load_ok(p, J, c.r, a, 16, kSiteGeneral)) lo[u] = ld_nc_stream(a);
        hi[u] = lo[u];
        dst[u] = J.out + 16 * kl;
        meta[u] = 0;  // kind 0: aligned vector, shift 0
        continue;
      }
      const uint64_t x = ((J.out >> 4) + kl) << 4;
      dst[u] = x;
      if (J.flags & kJobSmall) {
        meta[u] = 2u << 8;  // kind 2: bytes, small job
        continue;
      }
      unaligned_rank<MAXJ, MAXS>(c, J, x);
      if (x >= c.lo && x + 16 <= c.hi) {
        const uint64_t src = p.src[J.src0 + c.r] + (x - c.lo);
        const uint32_t s = static_cast<uint32_t>(src & 15u);
        const uint4* blk = reinterpret_cast<const uint4*>(src - s);
        if (s == 0) {
          if (load_ok(p, J, c.r, blk, 16, kSiteGeneral)) lo[u] = ld_nc_stream(blk);
          hi[u] = lo[u];
        } else {
          if (load_ok(p, J, c.r, blk, 16, kSiteGeneral)) lo[u] = ld_nc_cached(blk);
          if (load_ok(p, J, c.r, blk + 1, 16, kSiteGeneral)) hi[u] = ld_nc_cached(blk + 1);
        }
        meta[u] = s;  // kind 0
      } else {
        meta[u] = (1u << 8) | (c.r << 16);  // kind 1: bytes at a rank boundary
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      if (!dst[u]) continue;
      if (FLAT) {
        if (store_ok(p, p.job[job[u]], reinterpret_cast<void*>(dst[u]), 16, kSiteGeneral))
          st16(reinterpret_cast<uint4*>(dst[u]), lo[u]);
        continue;
      }
      const uint32_t kind = (meta[u] >> 8) & 0xFFu;
      if (kind == 0) {
        if (store_ok(p, p.job[job[u]], reinterpret_cast<void*>(dst[u]), 16, kSiteGeneral))
          st16(reinterpret_cast<uint4*>(dst[u]), realign16_sel(lo[u], hi[u], meta[u] & 15u));
      }
      else if (!FAST_EDGES)  // (the multi-CTA kernel has no registers to spare)
        copy_bytes(p, p.job[job[u]], dst[u], meta[u] >> 16, kind == 2);
      else if (kind == 2)
        copy_small_vector(p, p.job[job[u]], dst[u]);
      else
        copy_boundary(p, p.job[job[u]], dst[u], meta[u] >> 16);
    }
  }
}

// Kernel modes: kGeneral (any jobs), kFlat (all jobs 16-byte aligned),
// kFlat1 (one aligned job with fewer than 2^31 output vectors), kFlat1Staged
// (the same through shared memory), kManySplit (several jobs: the first
// flat_ctas CTAs stage the aligned jobs, the others stage and realign the
// rest).
enum Mode : int {
  kGeneral = 0,
  kFlat = 1,
  kFlat1 = 2,
  kFlat1Staged = 3,
  kManySplit = 4,
  kGeneral1Staged = 5,  // one unaligned job (>= kGatherSmallBytes per rank) through shared memory
  kGeneral1Warp = 6,    // the same, realigned across the lanes of a warp (32-bit indices)
};

template <int BLOCK, int UNROLL, int MODE, bool SINGLE = false, int MAXJ, int MAXS>
__device__ __forceinline__ void gather_mode(const GatherParams<MAXJ, MAXS>& p, uint64_t first,
                                            uint64_t step) {
  if constexpr (MODE == kFlat1 && MAXJ == 1)
    gather_tiles_flat1<BLOCK, UNROLL, uint32_t>(p, static_cast<uint32_t>(first),
                                                static_cast<uint32_t>(step));
  else if constexpr (MODE == kFlat1Staged && MAXJ == 1)
    gather_tiles_staged<BLOCK, kStagedVectors, kStagedStages>(p, static_cast<uint32_t>(first),
                                                              static_cast<uint32_t>(step));
  else if constexpr (MODE == kGeneral1Warp && MAXJ == 1) {
    // the last CTA copies the rank-boundary vectors, the others the rest
    if (first + 1 == step) {
      copy_boundaries<BLOCK>(p);
      return;
    }
    gather_tiles_warp_realign<BLOCK, kWarpRealignVectors>(p, static_cast<uint32_t>(first),
                                                          static_cast<uint32_t>(step - 1));
  }
  else if constexpr (MODE == kGeneral1Staged && MAXJ == 1) {
    // the last CTA copies the rank-boundary vectors, the others the rest
    if (first + 1 == step) {
      copy_boundaries<BLOCK>(p);
      return;
    }
    --step;
    const uint64_t span = p.total_vec * 16;  // output bytes from out rounded down to 16
    if (span < (1ull << 32) && p.job[0].bytes < (1ull << 32))
      gather_tiles_staged_realign<BLOCK, kRealignVectors, kRealignStages, uint32_t>(
          p, static_cast<uint32_t>(first), static_cast<uint32_t>(step));
    else
      gather_tiles_staged_realign<BLOCK, kRealignVectors, kRealignStages, uint64_t>(p, first, step);
  }
  else if constexpr (MODE == kManySplit) {
    // CTAs [0, fc): aligned jobs; [step - sc, step): the small jobs; [step -
    // sc - bc, step - sc): the rank-boundary vectors of the unaligned jobs
    // (warp realigning only); the rest: the other unaligned jobs
    const uint64_t fc = static_cast<uint64_t>(p.flat_ctas), sc = static_cast<uint64_t>(p.small_ctas);
    const uint64_t bc = static_cast<uint64_t>(p.bnd_ctas);
    if (first < fc)
      gather_tiles_staged_jobs<BLOCK, kSplitVectors, kSplitStages>(p, static_cast<uint32_t>(first),
                                                                   static_cast<uint32_t>(fc));
    else if (first + sc >= step) {
      if constexpr (MAXJ > 1) copy_small_jobs<BLOCK, kSmallSplit>(p, static_cast<uint32_t>(first + sc - step));
    }
    else if (first + sc + bc >= step)
      copy_boundaries_jobs<BLOCK>(p, static_cast<uint32_t>(first + sc + bc - step), static_cast<uint32_t>(bc));
    else if (p.realign_warp) {
      if (p.total_vec < (1ull << 28))  // 16 * vectors under 4 GiB
        gather_tiles_warp_realign_jobs<BLOCK, kSplitRealignVectors, uint32_t>(
            p, static_cast<uint32_t>(first - fc), static_cast<uint32_t>(step - fc - sc - bc),
            static_cast<uint32_t>(p.flat_vec), static_cast<uint32_t>(p.small_vec));
      else
        gather_tiles_warp_realign_jobs<BLOCK, kSplitRealignVectors, uint64_t>(
            p, static_cast<uint32_t>(first - fc), static_cast<uint32_t>(step - fc - sc - bc), p.flat_vec,
            p.small_vec);
    }
    else
      gather_tiles_staged_realign_jobs<BLOCK, kSplitRealignVectors, kSplitRealignStages>(
          p, static_cast<uint32_t>(first - fc), static_cast<uint32_t>(step - fc - sc), p.flat_vec, p.small_vec);
  } else
    gather_tiles<BLOCK, UNROLL, MODE != kGeneral, SINGLE>(p, first, step);
}

// One aligned job: the source bytes of output vectors [k, kend) (one
// segment per rank they cross) prefetched into L2.  Issued before the PDL
// wait, the HBM latency of the first tile overlaps the end of the previous
// kernel in the stream.
template <int MAXS>
__device__ __forceinline__ void prefetch_vectors(const GatherParams<1, MAXS>& p, uint64_t k,
                                                 uint64_t kend) {
  constexpr uint64_t kMaxVec = 2048;  // at most 32 KiB per prefetch instruction
  const uint64_t vp = p.job[0].bytes >> 4;
  kend = kend < p.total_vec ? kend : p.total_vec;
  while (k < kend) {
    const uint64_t r = k / vp;
    uint64_t seg = (r + 1) * vp < kend ? (r + 1) * vp : kend;
    seg = seg - k > kMaxVec ? k + kMaxVec : seg;
    const uint4* a = reinterpret_cast<const uint4*>(p.src[r]) + (k - r * vp);
    if (load_ok(p, p.job[0], static_cast<uint32_t>(r), a, (seg - k) * 16, kSitePrefetch))
      prefetch_l2(a, static_cast<uint32_t>((seg - k) * 16));
    k = seg;
  }
}

// One unaligned job: the source bytes of output vectors [k0, k1) (one span
// per rank they cross, widened to the 16-byte blocks holding its first and
// last byte, at most 32 KiB per prefetch instruction) prefetched into L2.
template <int MAXS>
__device__ __forceinline__ void prefetch_unaligned(const GatherParams<1, MAXS>& p, uint64_t k0,
                                                   uint64_t k1) {
  const GatherJob& J = p.job[0];
  const uint64_t xbase = J.out & ~static_cast<uint64_t>(15);
  const uint64_t out_end = J.out + static_cast<uint64_t>(p.P) * J.bytes;
  uint64_t y = max(xbase + 16 * k0, J.out);
  const uint64_t yend = min(xbase + 16 * k1, out_end);
  if (y >= yend) return;
  uint64_t r = (y - J.out) / J.bytes;
  while (y < yend && r < static_cast<uint64_t>(p.P)) {
    const uint64_t d = J.out + r * J.bytes;
    const uint64_t seg_end = min(yend, d + J.bytes);
    const uint64_t src = p.src[J.src0 + r];
    const uint64_t a0 = (src + (y - d)) & ~static_cast<uint64_t>(15);
    const uint64_t a1 = (src + (seg_end - d) + 15) & ~static_cast<uint64_t>(15);
    for (uint64_t c = a0; c < a1; c += 32768) {
      const uint64_t n = min(static_cast<uint64_t>(32768), a1 - c);
      if (load_ok(p, J, static_cast<uint32_t>(r), reinterpret_cast<const void*>(c), n, kSitePrefetch))
        prefetch_l2(reinterpret_cast<const void*>(c), static_cast<uint32_t>(n));
    }
    y = seg_end;
    ++r;
  }
}

// Multi-CTA gather: CTA c copies tiles c, c + gridDim.x, ...
template <int MAXJ, int MAXS, int MODE>
__global__ void __launch_bounds__(kGatherBlock, (MODE == kFlat1 || MODE == kFlat1Staged) ? 4
                                                : MODE == kGeneral1Staged ? 3 : MODE == kGeneral1Warp ? 2
                                                                                                     : 2)
    dc_gather_kernel(const __grid_constant__ GatherParams<MAXJ, MAXS> p) {
  if constexpr (MAXJ == 1 && (MODE == kFlat1 || MODE == kFlat1Staged)) {
    pdl_launch_dependents();
    if (threadIdx.x == 0) {  // the CTA's first p.prefetch tiles
      const uint64_t tile = static_cast<uint64_t>(p.tile_vec);
      uint64_t t = blockIdx.x;
      for (int i = 0; i < p.prefetch && t * tile < p.total_vec; ++i, t += gridDim.x)
        prefetch_vectors(p, t * tile, (t + 1) * tile);
    }
    pdl_wait();
  } else if constexpr (MAXJ == 1 && (MODE == kGeneral1Staged || MODE == kGeneral1Warp)) {
    // the first p.prefetch tiles of each tile CTA (all but the last CTA)
    // prefetched before the wait; dependents are let in after it (measured:
    // 8 x (256 KiB+1) back to back 2.87 us, 3.21 us with the trigger first,
    // 3.04 us without the prefetch)
    if (threadIdx.x == 0 && blockIdx.x + 1 < gridDim.x) {
      const uint64_t tile = static_cast<uint64_t>(p.tile_vec);
      uint64_t t = blockIdx.x;
      for (int i = 0; i < p.prefetch && t * tile < p.total_vec; ++i, t += gridDim.x - 1)
        prefetch_unaligned(p, t * tile, min((t + 1) * tile, p.total_vec));
    }
    pdl_wait();
    pdl_launch_dependents();
  } else {
    pdl_enter();
  }
  gather_mode<kGatherBlock, MODE == kGeneral ? kGatherUnrollGeneral : kGatherUnroll, MODE>(
      p, blockIdx.x, gridDim.x);
}

// Single-CTA gather for small outputs: one CTA copies everything.
template <int MAXJ, int MAXS, int MODE>
__global__ void __launch_bounds__(MODE == kGeneral ? kGatherSingleBlockGeneral : kGatherSingleBlock)
    dc_gather_single_kernel(const __grid_constant__ GatherParams<MAXJ, MAXS> p) {
  constexpr int kBlock = MODE == kGeneral ? kGatherSingleBlockGeneral : kGatherSingleBlock;
  if constexpr (MAXJ == 1 && MODE == kFlat1) {
    pdl_launch_dependents();
    if (p.prefetch && threadIdx.x < static_cast<unsigned>(p.P)) {
      // thread r: the start of rank r's payload (all of it below 32 KiB)
      const uint64_t vp = p.job[0].bytes >> 4;
      const uint64_t k = threadIdx.x * vp;
      prefetch_vectors(p, k, k + (vp < 2048 ? vp : 2048));
    }
    pdl_wait();
  } else {
    pdl_enter();
  }
  gather_mode<kBlock, MODE == kGeneral ? kGatherUnrollGeneral : kGatherUnroll, MODE, true>(p, 0, 1);
}

// The mode of a launch.  Jobs are ordered aligned first, so job 0 tells
// whether any job is aligned and flat_vec == total_vec whether all are.
template <int MAXJ, int MAXS>
int mode_of(const GatherParams<MAXJ, MAXS>& p) {
  const bool all_flat = p.flat_vec == p.total_vec;
  if (MAXJ > 1 && p.staged) return kManySplit;
  if (!all_flat) {
    if (MAXJ != 1 || !p.staged || (p.job[0].flags & kJobSmall)) return kGeneral;
    // the warp path uses 32-bit indices: outputs (from out rounded down to
    // 16) and ranks under 4 GiB
    const bool narrow = p.total_vec * 16 < (1ull << 32) && p.job[0].bytes < (1ull << 32);
    return p.realign_warp && narrow ? kGeneral1Warp : kGeneral1Staged;
  }
  if (MAXJ == 1 && p.total_vec < (1ull << 31)) return p.staged ? kFlat1Staged : kFlat1;
  return kFlat;
}

constexpr size_t staged_smem(int block) {
  return static_cast<size_t>(kStagedStages) * kStagedVectors * block * 16;
}

constexpr size_t split_smem(int block) {
  return static_cast<size_t>(kSplitStages) * kSplitVectors * block * 16;
}

constexpr size_t realign_smem(int block) {
  return static_cast<size_t>(kRealignStages) * kRealignVectors * 2 * block * 16;
}

template <int MODE>
constexpr size_t mode_smem() {
  return MODE == kFlat1Staged      ? staged_smem(kGatherBlock)
         : MODE == kManySplit      ? split_smem(kGatherBlock)
         : MODE == kGeneral1Staged ? realign_smem(kGatherBlock)
                                   : 0;
}

// Kernels that ask for more than 48 KB of dynamic shared memory must say so
// once per device (cudaFuncAttributeMaxDynamicSharedMemorySize).
template <int MAXJ, int MAXS, int MODE>
cudaError_t allow_smem() {
  constexpr size_t smem = mode_smem<MODE>();
  if constexpr (smem <= 48 * 1024) {
    return cudaSuccess;
  } else {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(dc_gather_kernel<MAXJ, MAXS, MODE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
}

template <int MAXJ, int MAXS, int MODE>
cudaError_t launch_mode(const GatherParams<MAXJ, MAXS>& p, int grid, bool single, bool pdl,
                        cudaStream_t s) {
  if (!single) {
    const cudaError_t e = allow_smem<MAXJ, MAXS, MODE>();
    if (e != cudaSuccess) return e;
  }
  if (single) {  // small outputs: staging buys nothing, use the register path
    constexpr int kMode = MODE == kFlat1Staged ? kFlat1
                          : (MODE == kManySplit || MODE == kGeneral1Staged || MODE == kGeneral1Warp) ? kGeneral
                                                                            : MODE;
    constexpr int block = kMode == kGeneral ? kGatherSingleBlockGeneral : kGatherSingleBlock;
    return launch_ex(dc_gather_single_kernel<MAXJ, MAXS, kMode>, 1, block, pdl, s, p);
  }
  return launch_ex(dc_gather_kernel<MAXJ, MAXS, MODE>, grid, kGatherBlock, pdl, s, p,
                   mode_smem<MODE>());
}

template <int MAXJ, int MAXS>
cudaError_t launch_impl(const GatherParams<MAXJ, MAXS>& p, int grid, bool single, bool pdl,
                        cudaStream_t s) {
  int mode = mode_of(p);
  // A split needs CTAs for each part that has work; otherwise one path for every CTA.
  if (mode == kManySplit) {
    const long long fc = p.flat_ctas, sc = p.small_ctas, rc = static_cast<long long>(grid) - fc - sc;
    if (single || fc < 0 || sc < 0 || rc < 0 || (p.flat_vec > 0 && fc < 1) ||
        (p.small_vec > p.flat_vec && rc < 1) || (p.total_vec > p.small_vec && sc < 1))
      mode = p.flat_vec == p.total_vec ? kFlat : kGeneral;
  }
  switch (mode) {
    case kGeneral: return launch_mode<MAXJ, MAXS, kGeneral>(p, grid, single, pdl, s);
    case kFlat: return launch_mode<MAXJ, MAXS, kFlat>(p, grid, single, pdl, s);
    case kManySplit:
      if constexpr (MAXJ > 1) return launch_mode<MAXJ, MAXS, kManySplit>(p, grid, single, pdl, s);
      return cudaErrorInvalidValue;
    case kGeneral1Staged:
      if constexpr (MAXJ == 1) {  // grid: at least one tile CTA and the boundary CTA
        if (!single && (grid < 2 || p.tile_vec < 1 || p.tile_vec > kGatherBlock * kRealignVectors))
          return cudaErrorInvalidValue;
        return launch_mode<MAXJ, MAXS, kGeneral1Staged>(p, grid, single, pdl, s);
      }
      return cudaErrorInvalidValue;
    case kGeneral1Warp:
      if constexpr (MAXJ == 1) {  // grid: at least one tile CTA and the boundary CTA
        if (!single && (grid < 2 || p.tile_vec < 1 || p.tile_vec > kGatherBlock * kWarpRealignVectors))
          return cudaErrorInvalidValue;
        return launch_mode<MAXJ, MAXS, kGeneral1Warp>(p, grid, single, pdl, s);
      }
      return cudaErrorInvalidValue;
    case kFlat1:
      if constexpr (MAXJ == 1) return launch_mode<MAXJ, MAXS, kFlat1>(p, grid, single, pdl, s);
      return cudaErrorInvalidValue;
    default:
      if constexpr (MAXJ == 1) {
        if (!single && (p.tile_vec < 1 || p.tile_vec > kGatherBlock * kStagedVectors))
          return cudaErrorInvalidValue;
        return launch_mode<MAXJ, MAXS, kFlat1Staged>(p, grid, single, pdl, s);
      }
      return cudaErrorInvalidValue;
  }
}

template <int MAXJ, int MAXS>
int occupancy_impl(int mode) {
  int n = 0;
  cudaError_t e;
  if (mode == kGeneral)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dc_gather_kernel<MAXJ, MAXS, kGeneral>,
                                                      kGatherBlock, 0);
  else if (mode == kFlat || (MAXJ != 1 && mode != kManySplit) || (MAXJ != 1 && mode == kGeneral1Staged))
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dc_gather_kernel<MAXJ, MAXS, kFlat>,
                                                      kGatherBlock, 0);
  else if (mode == kGeneral1Warp && MAXJ == 1) {
    constexpr int kM = MAXJ == 1 ? kGeneral1Warp : kGeneral;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dc_gather_kernel<MAXJ, MAXS, kM>, kGatherBlock, 0);
  } else if (mode == kGeneral1Staged && MAXJ == 1) {
    constexpr int kM = MAXJ == 1 ? kGeneral1Staged : kGeneral;
    e = allow_smem<MAXJ, MAXS, kM>();
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dc_gather_kernel<MAXJ, MAXS, kM>,
                                                        kGatherBlock, mode_smem<kM>());
  } else if (mode == kManySplit && MAXJ > 1) {
    constexpr int kM = MAXJ == 1 ? kFlat : kManySplit;
    e = allow_smem<MAXJ, MAXS, kM>();
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dc_gather_kernel<MAXJ, MAXS, kM>,
                                                        kGatherBlock, mode_smem<kM>());
  }
  else if (mode == kFlat1)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &n, dc_gather_kernel<MAXJ, MAXS, MAXJ == 1 ? kFlat1 : kFlat>, kGatherBlock, 0);
  else
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &n, dc_gather_kernel<MAXJ, MAXS, MAXJ == 1 ? kFlat1Staged : kFlat>, kGatherBlock,
        MAXJ == 1 ? staged_smem(kGatherBlock) : 0);
  if (e != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_gather(const GatherParams1& p, int grid, bool single, bool pdl, cudaStream_t s) {
  return launch_impl(p, grid, single, pdl, s);
}
cudaError_t launch_gather(const GatherParamsS& p, int grid, bool single, bool pdl, cudaStream_t s) {
  return launch_impl(p, grid, single, pdl, s);
}
cudaError_t launch_gather(const GatherParamsL& p, int grid, bool single, bool pdl, cudaStream_t s) {
  return launch_impl(p, grid, single, pdl, s);
}

int gather_ctas_per_sm(int which, int mode) {
  switch (which) {
    case 0: return occupancy_impl<1, kMaxRanks>(mode);
    case 1: return occupancy_impl<kManySmallTensors, kManySmallSegments>(mode);
    default: return occupancy_impl<kManyMaxTensors, kManyMaxSegments>(mode);
  }
}

DC_BOUNDS_READER(take_bounds_gather)

int gather_mode_of(const GatherParams1& p) { return mode_of(p); }
int gather_mode_of(const GatherParamsS& p) { return mode_of(p); }
int gather_mode_of(const GatherParamsL& p) { return mode_of(p); }

}  // namespace dc
