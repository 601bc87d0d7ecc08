// dc_bulk.cu -- the 16-byte aligned rank-ordered gather on the TMA engine.
//
// "perf(cuda): vectorize the deterministic all-gather copy and right-size its
// single-block path" (RL-Kernel PR 491), section "What": when the output, the
// size and every payload are 16-byte aligned, the gathered output is one flat
// copy across all ranks, out[r*B + j] = src_r[j].
//
// Design on one GB300.  The thread-per-16-byte-vector copies spend a few
// instructions on every vector (address, load or cp.async, shared-memory
// read, store); at 4 MiB per rank that keeps them issue- and latency-bound
// well below the HBM rate.  Here the copy is made of 1-D bulk copies, which
// move whole chunks per instruction:
//  * The output is cut into chunks of `chunk` bytes (a multiple of 16; sized
//    by the planner so that every CTA gets the same number of equal chunks).
//    CTA c takes chunks c, c + G, c + 2G, ... so that all CTAs sweep the
//    buffers together.
//  * One thread per CTA drives a ring of S shared-memory stages, each with
//    an mbarrier.  A chunk is loaded by one bulk copy per rank piece it
//    covers (cp.async.bulk global -> shared, completing on the stage's
//    mbarrier with its byte count); when the stage's phase completes, one
//    bulk store (cp.async.bulk shared -> global, a bulk group) writes it to
//    the output, and the stage is refilled with the chunk S steps ahead once
//    that store has read it (cp.async.bulk.wait_group.read).  S - 1 chunks'
//    loads stay in flight per CTA.
//  * Every mbarrier wait is bounded: at most `wait_ns` of the global timer
//    (and a poll count).  A wait that runs out records kFaultBulkWait in a
//    device fault word (read and cleared by dc_check_device), waits again,
//    with the same bound, for the CTA's other loads in flight, waits until
//    its stores have read shared memory, and returns.  A failure is
//    therefore reported, never a hang.
//  * Programmatic dependent launch: the CTA lets the next kernel of the
//    stream launch at once, prefetches the sources of its first `prefetch`
//    chunks into L2, and waits for the previous kernel before its first bulk
//    load; as it issues each chunk's load it prefetches the chunk `prefetch`
//    steps ahead.
//  * No tensor map, no cluster and no multicast: sources and output are
//    buffers of this GPU's own memory.
#include <atomic>

#include "dc_device.cuh"
#include "dc_internal.h"
#include "dc_tma.cuh"

namespace dc {
namespace {

using namespace tma;

// Fault bits of the kernels in this file (kFault*), sticky until
// take_bulk_faults reads and clears them.
__device__ unsigned int g_bulk_fault_bits;

// Output bytes [o0, o0 + len) of the gather come from rank r = o / B at
// offset o - r*B, one piece per rank they cross: f(o, piece bytes, rank's
// source address) for each piece whose source range passes the bounds check
// of the checked build (the rank's whole source).
enum : uint32_t { kSiteBulkLoad = 300, kSiteBulkStore = 301, kSiteBulkPrefetch = 302 };
template <class F>
__device__ __forceinline__ void for_each_piece(const BulkParams& p, uint64_t o0, uint64_t len, uint32_t site,
                                               F f) {
  const uint64_t B = p.bytes, end = o0 + len;
  uint64_t r = o0 / B, o = o0;
  while (o < end) {
    const uint64_t rend = min((r + 1) * B, end);
    const uint8_t* a = reinterpret_cast<const uint8_t*>(p.src[r]) + (o - r * B);
    if (in_bounds(a, rend - o, p.src[r], p.src[r] + B, site)) f(o, rend - o, a);
    o = rend;
    ++r;
  }
}

__global__ void __launch_bounds__(32) dc_gather_bulk_kernel(const __grid_constant__ BulkParams p) {
  pdl_launch_dependents();
  if (threadIdx.x != 0) return;
  extern __shared__ __align__(128) uint8_t bulk_smem[];  // [stages][chunk], then the mbarriers
  const uint32_t S = static_cast<uint32_t>(p.stages);
  const uint64_t chunk = p.chunk, total = p.total;
  const uint64_t nchunks = (total + chunk - 1) / chunk;
  const uint64_t c0 = blockIdx.x, step = gridDim.x, cend = nchunks;  // chunks c0, c0 + step, ...
  const uint32_t buf = static_cast<uint32_t>(__cvta_generic_to_shared(bulk_smem));
  const uint32_t bars = buf + S * static_cast<uint32_t>(chunk);
  for (uint32_t k = 0; k < S; ++k) mbar_init(bars + 8u * k, 1);
  mbar_init_fence();
  // L2 prefetch: the CTA's first p.prefetch chunks before the wait, then, as
  // each chunk's load is issued, the chunk p.prefetch steps ahead of it
  const uint64_t pf = static_cast<uint64_t>(p.prefetch);
  auto prefetch_chunk = [&](uint64_t c) {
    if (c >= cend) return;
    for_each_piece(p, c * chunk, min(chunk, total - c * chunk), kSiteBulkPrefetch,
                   [](uint64_t, uint64_t n, const uint8_t* a) {
      for (uint64_t q = 0; q < n; q += 32768)
        prefetch_l2(a + q, static_cast<uint32_t>(min(n - q, static_cast<uint64_t>(32768))));
    });
  };
  for (uint64_t q = 0; q < pf; ++q) prefetch_chunk(c0 + q * step);
  pdl_wait();

  uint32_t inflight = 0;  // bit k: stage k has loads issued and not yet waited for
  auto issue = [&](uint32_t k, uint64_t c) {
    const uint64_t o0 = c * chunk, len = min(chunk, total - o0);
    const uint32_t bar = bars + 8u * k, dst = buf + k * static_cast<uint32_t>(chunk);
    // (test only: announce 16 bytes that never come, so that this wait runs out)
    const uint32_t extra = (p.test_flags & kBulkTestShortTx) && c == c0 ? 16u : 0u;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(len) + extra);
    for_each_piece(p, o0, len, kSiteBulkLoad, [&](uint64_t o, uint64_t n, const uint8_t* a) {
      bulk_load(dst + static_cast<uint32_t>(o - o0), a, static_cast<uint32_t>(n), bar);
    });
    inflight |= 1u << k;
    if (pf) prefetch_chunk(c + pf * step);
  };
  {
    uint64_t c = c0;
    for (uint32_t k = 0; k < S && c < cend; ++k, c += step) issue(k, c);
  }
  uint32_t phase = 0;  // bit k: parity of stage k's next phase
  uint32_t k = 0, kprev = S - 1;
  bool ok = true;
  uint64_t i = 0;
  for (uint64_t c = c0; c < cend; c += step, ++i) {
    const uint32_t bar = bars + 8u * k;
    if (!mbar_wait_bounded(bar, (phase >> k) & 1u, p.wait_ns)) {
      inflight &= ~(1u << k);  // already waited for once
      ok = false;
      break;
    }
    phase ^= 1u << k;
    inflight &= ~(1u << k);
    fence_proxy_async_smem();
    const uint64_t o0 = c * chunk, len = min(chunk, total - o0);
    uint8_t* d = reinterpret_cast<uint8_t*>(p.out) + o0;
    if (in_bounds(d, len, p.out, p.out + total, kSiteBulkStore))
      bulk_store(d, buf + k * static_cast<uint32_t>(chunk), static_cast<uint32_t>(len));
    bulk_commit();
    if (S == 1) {  // one stage: refill it once its store has read it
      if (c + step < cend) {
        bulk_wait_read<0>();
        issue(0, c + step);
      }
    } else if (i > 0) {  // refill the stage drained one step ago with the chunk S - 1 steps ahead
      const uint64_t cn = c + (S - 1) * step;
      if (cn < cend) {
        bulk_wait_read<1>();
        issue(kprev, cn);
      }
    }
    kprev = k;
    k = (k + 1 == S) ? 0 : k + 1;
  }
  if (!ok) {
    atomicOr(&g_bulk_fault_bits, kFaultBulkWait);
    for (uint32_t q = 0; q < S; ++q)
      if ((inflight >> q) & 1u) mbar_wait_bounded(bars + 8u * q, (phase >> q) & 1u, p.wait_ns);
  }
  bulk_wait_read<0>();  // the stores have read shared memory; their writes complete with the grid
}

}  // namespace

size_t bulk_smem_bytes(uint64_t chunk, int stages) {
  return static_cast<size_t>(stages) * (static_cast<size_t>(chunk) + 8);
}

cudaError_t launch_gather_bulk(const BulkParams& p, int grid, bool pdl, cudaStream_t s) {
  const size_t smem = bulk_smem_bytes(p.chunk, p.stages);
  if (grid < 1 || p.stages < 1 || p.stages > 32 || p.chunk < 16 || (p.chunk & 15u) || smem > kBulkMaxSmem ||
      p.bytes == 0 || (p.bytes & 15u) || p.total != p.bytes * static_cast<uint64_t>(p.P))
    return cudaErrorInvalidValue;
  static std::atomic<uint64_t> done{0};  // devices on which the kernel may use kBulkMaxSmem
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(dc_gather_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kBulkMaxSmem));
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_release);
  }
  return launch_ex(dc_gather_bulk_kernel, grid, 32, pdl, s, p, smem);
}

DC_BOUNDS_READER(take_bounds_bulk)

cudaError_t take_bulk_faults(uint32_t* bits) {
  *bits = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_bulk_fault_bits, sizeof v);
  if (e != cudaSuccess) return e;
  if (v) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_bulk_fault_bits, &zero, sizeof zero);
  }
  *bits = v;
  return e;
}

}  // namespace dc
