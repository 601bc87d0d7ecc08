// dc_fused.cu -- the staged all-gather protocol of a multi-rank deterministic
// collective (stage -> gather -> complete), with every wait bounded.
//
// "perf(cuda): vectorize the deterministic all-gather copy and right-size its
// single-block path" (RL-Kernel PR 491) describes the deployment behind the
// copy: a backend named cuda_ipc_fixed_tree whose ranks exchange payloads
// through staging buffers that their peers map and read, in a CUDA-graph-safe
// fused protocol of three steps -- each rank stages its payload, gathers its
// peers' staged payloads, and completes, after which its staging buffer may be
// reused (author's replies).  The page leaves open that a failed launch leaves
// that protocol pending with no abort path, and that when a rank dies its
// peers wait until the process-group timeout (section "Not in this PR" and the
// review threads on the pending state and on the distributed test).
//
// Here the P ranks are groups of CTAs of ONE cooperative launch on one GPU:
// the cooperative launch makes every CTA of the grid resident at once, so a
// CTA may wait for another without deadlock.  Rank r owns an input, a staging
// buffer and an output; its B bytes are cut into G chunks, and CTA (r, c)
// handles chunk c of rank r:
//   stage:    in_r[chunk c] -> staging_r[chunk c]; then staged[r][c] = epoch
//             (release store, after a device-scope fence by every thread);
//   gather:   wait until staged[q][c] == epoch for every rank q (acquire
//             loads), then staging_q[chunk c] -> out_r[q*B + chunk c] for
//             every q: by default one thread streams the chunks through the
//             TMA engine (gather_tma: bulk loads into a shared-memory ring,
//             bulk stores out of it), else every thread copies 16-byte
//             vectors (loads through L2 only: staging_q is written by other
//             CTAs);
//   complete: done[r][c] = epoch, then wait until done[q][c] == epoch for
//             every q: chunk c of staging_r has been read by every rank and
//             may be overwritten by the next epoch.
// The flags live in a caller-owned workspace of P x kFusedMaxChunks x 2
// words, zero before the first call; each call carries a new epoch (1, 2,
// 3, ...), so no flag is ever reset between calls.  Every wait is bounded by
// wait_ns of the global timer and a poll count.  A wait that runs out records
// the first fault (phase, waiting rank, awaited rank, chunk, epoch) in a
// device fault word read by dc_check_device, and the CTA returns: a rank that
// never arrives makes its peers report DC_ERR_TIMEOUT within the bound
// instead of hanging.  The caller then clears the workspace and starts again
// at epoch 1 (dc_fused_reset): that is the abort path.
#include <atomic>
#include <mutex>

#include "dc_device.cuh"
#include "dc_internal.h"
#include "dc_tma.cuh"

namespace dc {
namespace {

// First fault of a fused launch: [0] kFaultFusedWait bits, [1] phase << 24 |
// waiting rank << 12 | awaited rank, [2] chunk, [3] epoch.  Sticky until
// take_fused_faults reads and clears it.
__device__ unsigned int g_fused_fault[4];

using tma::global_ns;

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16-byte load through L2 only (no L1 line that could hold an older epoch's
// bytes of a staging buffer).
__device__ __forceinline__ uint4 ld_cg16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Waits until *f == want, for at most limit_ns of the global timer and at
// most 2^24 polls.  False: it ran out.
__device__ __forceinline__ bool wait_flag(const uint32_t* f, uint32_t want, uint64_t limit_ns) {
  if (ld_acquire_u32(f) == want) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 24); ++i) {
    __nanosleep(64);
    if (ld_acquire_u32(f) == want) return true;
    if (global_ns() - t0 >= limit_ns) return false;
  }
  return false;
}

__device__ __forceinline__ void record_fault(uint32_t phase, uint32_t rank, uint32_t peer, uint32_t chunk,
                                             uint32_t epoch) {
  if (atomicCAS(&g_fused_fault[0], 0u, kFaultFusedWait) == 0u) {
    g_fused_fault[1] = (phase << 24) | (rank << 12) | peer;
    g_fused_fault[2] = chunk;
    g_fused_fault[3] = epoch;
    __threadfence();
  }
}

// Sites of the checked build's bounds checks (in_bounds).
enum : uint32_t { kSiteFusedStage = 400, kSiteFusedGather = 401, kSiteFusedFlag = 402 };

// n bytes (a multiple of 16; both pointers 16-byte aligned) copied by the
// CTA's threads, U 16-byte vectors in flight per thread.  Checked build:
// loads inside [slo, shi), stores inside [dlo, dhi).
template <bool THROUGH_L2, int U>
__device__ __forceinline__ void copy_chunk(const uint8_t* src, uint8_t* dst, uint64_t n, uint64_t slo,
                                           uint64_t shi, uint64_t dlo, uint64_t dhi, uint32_t site) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  const uint64_t nv = n >> 4;
  for (uint64_t i = threadIdx.x; i < nv; i += static_cast<uint64_t>(U) * kFusedBlock) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t k = i + static_cast<uint64_t>(u) * kFusedBlock;
      if (k < nv && in_bounds(s + k, 16, slo, shi, site)) v[u] = THROUGH_L2 ? ld_cg16(s + k) : ld_stream(s + k);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t k = i + static_cast<uint64_t>(u) * kFusedBlock;
      if (k < nv && in_bounds(d + k, 16, dlo, dhi, site)) st16(d + k, v[u]);
    }
  }
}

// The gather step on the TMA engine: thread 0 streams the P staged chunks
// (peers in the order q0, q0+1, ...) through a ring of p.stages shared-memory
// stages of p.sub bytes: each piece is one bulk load (staging_q -> stage,
// completing on the stage's mbarrier) and one bulk store (stage -> out_r),
// with p.stages - 1 pieces' loads in flight; the stores drain through the
// TMA engine instead of the load-store units.  Every mbarrier wait is
// bounded; one that runs out records the fault (phase 3), waits (bounded)
// for the loads still in flight and returns false.  True: every load has
// landed, so the staging chunks have been read.
__device__ __forceinline__ bool gather_tma(const FusedParams& p, uint32_t r, uint32_t c, uint32_t q0, uint64_t lo,
                                           uint64_t n) {
  using namespace tma;
  extern __shared__ __align__(128) uint8_t fused_smem[];  // [stages][sub], then the mbarriers
  const uint32_t P = static_cast<uint32_t>(p.P), S = static_cast<uint32_t>(p.stages);
  const uint64_t sub = p.sub, B = p.bytes;
  const uint32_t buf = static_cast<uint32_t>(__cvta_generic_to_shared(fused_smem));
  const uint32_t bars = buf + S * static_cast<uint32_t>(sub);
  for (uint32_t k = 0; k < S; ++k) mbar_init(bars + 8u * k, 1);
  mbar_init_fence();
  // the staged bytes were published by other CTAs (release/acquire on the
  // flags, generic proxy); the bulk loads below read them through the async proxy
  fence_proxy_async_global();
  const uint64_t per = (n + sub - 1) / sub, items = per * P;
  auto piece = [&](uint64_t i, uint32_t& q, uint64_t& off) {
    const uint64_t pi = i / per;
    q = q0 + static_cast<uint32_t>(pi);
    if (q >= P) q -= P;
    off = (i - pi * per) * sub;
  };
  uint32_t inflight = 0, phase = 0;
  auto issue = [&](uint32_t k, uint64_t i) {
    uint32_t q;
    uint64_t off;
    piece(i, q, off);
    const uint32_t len = static_cast<uint32_t>(min(sub, n - off));
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.staging[q]) + lo + off;
    const bool ok = in_bounds(src, len, p.staging[q], p.staging[q] + B, kSiteFusedGather);
    mbar_arrive_expect_tx(bars + 8u * k, ok ? len : 0u);
    if (ok) bulk_load(buf + k * static_cast<uint32_t>(sub), src, len, bars + 8u * k);
    inflight |= 1u << k;
  };
  for (uint32_t k = 0; k < S && k < items; ++k) issue(k, k);
  bool ok = true;
  uint32_t k = 0, kprev = S - 1;
  for (uint64_t i = 0; i < items; ++i) {
    if (!mbar_wait_bounded(bars + 8u * k, (phase >> k) & 1u, p.wait_ns)) {
      uint32_t q;
      uint64_t off;
      piece(i, q, off);
      record_fault(3, r, q, c, p.epoch);
      inflight &= ~(1u << k);  // already waited for once
      ok = false;
      break;
    }
    phase ^= 1u << k;
    inflight &= ~(1u << k);
    fence_proxy_async_smem();
    uint32_t q;
    uint64_t off;
    piece(i, q, off);
    const uint32_t len = static_cast<uint32_t>(min(sub, n - off));
    uint8_t* dst = reinterpret_cast<uint8_t*>(p.out[r]) + static_cast<uint64_t>(q) * B + lo + off;
    if (in_bounds(dst, len, p.out[r], p.out[r] + P * B, kSiteFusedGather))
      bulk_store(dst, buf + k * static_cast<uint32_t>(sub), len);
    bulk_commit();
    if (S == 1) {  // one stage: refill it once its store has read it
      if (i + 1 < items) {
        bulk_wait_read<0>();
        issue(0, i + 1);
      }
    } else if (i > 0 && i + S - 1 < items) {  // refill the stage drained one step ago
      bulk_wait_read<1>();
      issue(kprev, i + S - 1);
    }
    kprev = k;
    k = (k + 1 == S) ? 0 : k + 1;
  }
  if (!ok)
    for (uint32_t q = 0; q < S; ++q)
      if ((inflight >> q) & 1u) mbar_wait_bounded(bars + 8u * q, (phase >> q) & 1u, p.wait_ns);
  bulk_wait_read<0>();  // the stores have read the stages; their writes complete with the grid
  return ok;
}

__global__ void __launch_bounds__(kFusedBlock) dc_fused_gather_kernel(const __grid_constant__ FusedParams p) {
  __shared__ int s_ok[1];
  const uint32_t P = static_cast<uint32_t>(p.P), G = static_cast<uint32_t>(p.G);
  const uint32_t r = blockIdx.x / G, c = blockIdx.x % G;
  if (r >= P) return;
  if ((p.absent >> r) & 1ull) return;  // (test only: a rank that never arrives)
  uint32_t* staged = reinterpret_cast<uint32_t*>(p.ws);
  uint32_t* done = staged + static_cast<uint64_t>(P) * kFusedMaxChunks;
  const uint64_t lo = static_cast<uint64_t>(c) * p.chunk;
  const uint64_t n = lo < p.bytes ? min(p.chunk, p.bytes - lo) : 0;
  const uint32_t epoch = p.epoch;

  // stage
  copy_chunk<false, 8>(reinterpret_cast<const uint8_t*>(p.in[r]) + lo, reinterpret_cast<uint8_t*>(p.staging[r]) + lo,
                    n, p.in[r], p.in[r] + p.bytes, p.staging[r], p.staging[r] + p.bytes, kSiteFusedStage);
  __threadfence();
  __syncthreads();
  const uint64_t ws_lo = p.ws, ws_hi = p.ws + fused_workspace_bytes(static_cast<int>(P));
  if (threadIdx.x == 0 && in_bounds(&staged[r * kFusedMaxChunks + c], 4, ws_lo, ws_hi, kSiteFusedFlag))
    st_release_u32(&staged[r * kFusedMaxChunks + c], epoch);

  // gather: thread 0 waits until every rank has published chunk c, then the
  // CTA copies the P staged chunks without a barrier between them (a barrier
  // per peer drained the loads in flight each time).  Peers are taken in the
  // order c, c+1, ... (mod P), the same for every rank: the P CTAs of chunk c
  // read staging_q's chunk at about the same time, while it is in L2 (in a
  // per-rank order the P reads of one chunk spread over the whole gather and
  // the output traffic evicted the chunk in between).
  const uint32_t q0 = c % P;
  if (threadIdx.x == 0) {
    bool ok = true;
    for (uint32_t i = 0; i < P && ok; ++i) {
      const uint32_t q = q0 + i < P ? q0 + i : q0 + i - P;
      ok = in_bounds(&staged[q * kFusedMaxChunks + c], 4, ws_lo, ws_hi, kSiteFusedFlag) &&
           wait_flag(&staged[q * kFusedMaxChunks + c], epoch, p.wait_ns);
      if (!ok) record_fault(1, r, q, c, epoch);
    }
    __threadfence();
    s_ok[0] = ok;
  }
  __syncthreads();
  if (!s_ok[0]) return;
  if (p.tma) {
    // one thread drives the TMA ring; the others are done
    if (threadIdx.x != 0) return;
    if (!gather_tma(p, r, c, q0, lo, n)) return;  // fault recorded; no completion to publish
  } else {
    for (uint32_t i = 0; i < P; ++i) {
      const uint32_t q = q0 + i < P ? q0 + i : q0 + i - P;
      copy_chunk<true, 8>(reinterpret_cast<const uint8_t*>(p.staging[q]) + lo,
                          reinterpret_cast<uint8_t*>(p.out[r]) + static_cast<uint64_t>(q) * p.bytes + lo, n,
                          p.staging[q], p.staging[q] + p.bytes, p.out[r], p.out[r] + P * p.bytes,
                          kSiteFusedGather);
    }
    __threadfence();
    __syncthreads();
  }

  // complete
  if (threadIdx.x == 0) {
    if (in_bounds(&done[r * kFusedMaxChunks + c], 4, ws_lo, ws_hi, kSiteFusedFlag))
      st_release_u32(&done[r * kFusedMaxChunks + c], epoch);
    for (uint32_t q = 0; q < P; ++q)
      if (!in_bounds(&done[q * kFusedMaxChunks + c], 4, ws_lo, ws_hi, kSiteFusedFlag) ||
          !wait_flag(&done[q * kFusedMaxChunks + c], epoch, p.wait_ns)) {
        record_fault(2, r, q, c, epoch);
        break;
      }
  }
}

}  // namespace

// Lets the kernel use `smem` bytes of dynamic shared memory (the TMA ring
// needs more than the default 48 KB; the kernel's own static shared memory
// counts against the same limit, so the attribute is raised to what a launch
// asks for, per device, never lowered).
cudaError_t allow_fused_smem(size_t smem) {
  if (smem <= 48u * 1024u) return cudaSuccess;
  constexpr int kDevices = 64;
  static std::atomic<size_t> allowed[kDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
  if (allowed[dev].load(std::memory_order_acquire) >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(dc_fused_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  size_t cur = allowed[dev].load(std::memory_order_relaxed);
  while (cur < smem && !allowed[dev].compare_exchange_weak(cur, smem)) {
  }
  return cudaSuccess;
}

int fused_ctas_per_sm(size_t smem) {
  int n = 0;
  if (allow_fused_smem(smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dc_fused_gather_kernel, kFusedBlock, smem) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n > 0 ? n : 1;
}

cudaError_t launch_fused_gather(const FusedParams& p, cudaStream_t s) {
  if (p.P < 1 || p.P > kMaxRanks || p.G < 1 || p.G > kFusedMaxChunks || (p.chunk & 15u) || (p.bytes & 15u) ||
      p.epoch == 0 || static_cast<uint64_t>(p.G) * p.chunk < p.bytes)
    return cudaErrorInvalidValue;
  const size_t smem = fused_smem_bytes(p.tma, p.stages, p.sub);
  if (p.tma && (p.stages < 1 || p.stages > 32 || p.sub < 16 || (p.sub & 15u) || smem > kFusedMaxSmem))
    return cudaErrorInvalidValue;
  cudaError_t e = allow_fused_smem(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.P * p.G));
  cfg.blockDim = dim3(kFusedBlock);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dc_fused_gather_kernel, p);
}

// ------------------------------------------------ allocation-free form ---
// Scratch of dc_fused_all_gather_static, for callers that cannot allocate
// device memory: the epoch flags of kMaxRanks ranks (64 KiB), then
// kFusedStaticStagingBytes (16 MiB) of staging buffers.  The array is part of
// this file's device code, so every GPU that loads it holds these bytes until
// the process exits; every call shares them.  In host code the name
// g_fused_scratch only stands in for the array: its device address comes from
// cudaGetSymbolAddress, once per device (static_scratch below).
constexpr size_t kFusedStaticFlagBytes = fused_workspace_bytes(kMaxRanks);
static __device__ __align__(256) unsigned char g_fused_scratch[kFusedStaticFlagBytes + kFusedStaticStagingBytes];

namespace {

// The device address of g_fused_scratch on the current device, looked up on
// the first call made with that device current and remembered.
cudaError_t static_scratch(unsigned char** ptr) {
  constexpr int kDevices = 64;
  static std::mutex mu;
  static unsigned char* addr[kDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fused_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<unsigned char*>(p);
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_fused_gather_static(FusedParams p, cudaStream_t s) {
  const uint64_t stride = fused_static_stride(p.bytes);
  if (p.P < 1 || p.P > kMaxRanks || stride * static_cast<uint64_t>(p.P) > kFusedStaticStagingBytes)
    return cudaErrorInvalidValue;
  unsigned char* base = nullptr;
  cudaError_t e = static_scratch(&base);
  if (e != cudaSuccess) return e;
  // the flags must start at zero: the previous call left its epoch in them
  e = cudaMemsetAsync(base, 0, fused_workspace_bytes(p.P), s);
  if (e != cudaSuccess) return e;
  p.ws = reinterpret_cast<uint64_t>(base);
  for (int r = 0; r < p.P; ++r)
    p.staging[r] = reinterpret_cast<uint64_t>(base + kFusedStaticFlagBytes + stride * static_cast<uint64_t>(r));
  p.epoch = 1;
  return launch_fused_gather(p, s);
}

DC_BOUNDS_READER(take_bounds_fused)

cudaError_t take_fused_faults(uint32_t* info) {
  for (int i = 0; i < 4; ++i) info[i] = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned int v[4] = {0, 0, 0, 0};
  e = cudaMemcpyFromSymbol(v, g_fused_fault, sizeof v);
  if (e != cudaSuccess) return e;
  if (v[0]) {
    const unsigned int zero[4] = {0, 0, 0, 0};
    e = cudaMemcpyToSymbol(g_fused_fault, zero, sizeof zero);
  }
  for (int i = 0; i < 4; ++i) info[i] = v[i];
  return e;
}

}  // namespace dc
