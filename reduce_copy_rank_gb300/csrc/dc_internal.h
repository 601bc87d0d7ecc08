// dc_internal.h -- definitions shared by the host planner (dc_api.cu) and the
// kernels (dc_gather.cu, dc_reduce.cuh and its per-type units, dc_delay.cu).
// Not part of the public C ABI.
//
// Everything a kernel needs travels by value in one parameter block, so a
// launch allocates nothing, reads no host memory after it is enqueued and can
// be captured in a CUDA graph.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dc {

constexpr int kMaxRanks = 64;            // P limit (pointer tables stay small)
constexpr int kManyMaxTensors = 256;     // all_gather_many: tensors per call
constexpr int kManyMaxSegments = 1024;   // all_gather_many: tensors x ranks
constexpr int kManySmallTensors = 16;    // the small parameter block of all_gather_many
constexpr int kManySmallSegments = 128;

// Threads per CTA of each kernel family.
constexpr int kGatherBlock = 512;
constexpr int kGatherSingleBlock = 1024;       // aligned (flat) jobs only
constexpr int kGatherSingleBlockGeneral = 512;  // any job: the realigning path needs registers
constexpr int kGatherUnroll = 4;         // 16-byte vectors in flight per thread (aligned)
constexpr int kGatherUnrollGeneral = 2;  // realigned vectors (up to two loads each) per thread
// Shared-memory staged aligned copy: kStagedStages ring slots of
// kStagedVectors 16-byte vectors per thread (2 x 3 x 512 x 16 B = 48 KB per
// CTA, four CTAs = 192 KB in flight per SM, no registers held).
constexpr int kStagedStages = 2;
constexpr int kStagedVectors = 3;
// all_gather_many with 16-byte aligned jobs: the aligned jobs are copied by
// the first part of the grid through a deeper ring (the kernel also carries
// the realigning path, so two CTAs fit per SM: 2 x 96 KB in flight).
constexpr int kSplitStages = 3;
constexpr int kSplitVectors = 4;
// ... and the unaligned jobs by the rest of the grid through a ring of the
// same size: 3 slots x 2 vectors x 2 source blocks.
constexpr int kSplitRealignStages = 3;
constexpr int kSplitRealignVectors = 2;
// One unaligned job staged through shared memory: per thread kRealignStages
// slots of kRealignVectors output vectors, each with the two aligned source
// blocks it is cut from (2 x 2 x 2 x 512 x 16 B = 64 KB per CTA, three CTAs
// per SM).
constexpr int kRealignStages = 2;
constexpr int kRealignVectors = 2;
// One unaligned job realigned across a warp (mode 6): output vectors in
// flight per thread, loaded straight into registers.
constexpr int kWarpRealignVectors = 4;
constexpr int kReduceBlock = 256;
constexpr int kReduceSingleBlock = 512;
constexpr int kReduceUnroll = 2;         // 8-element groups in flight per thread (P = 8 or any P)
// Groups in flight per thread of the kernel compiled for P = pt (0: any P):
// 16 rank loads in flight for P = 2, 4 and 8.
__host__ __device__ constexpr int reduce_unroll(int pt) {
  return pt == 2 ? 8 : pt == 4 ? 4 : kReduceUnroll;
}
// The staged realigning all_reduce (one job, P = 2, 4 or 8): ring stages,
// and per stage, rank and warp of kReduceBlock threads 33 blocks of 16 bytes
// (P = 8: 3 x 8 x 8 x 33 x 16 B = 99 KB per CTA, two CTAs per SM).
constexpr int kRealignReduceStages = 3;
__host__ __device__ constexpr size_t realign_reduce_smem(int pt) {
  return static_cast<size_t>(kRealignReduceStages) * pt * (kReduceBlock / 32) * 33 * 16;
}
// The compile-time rank counts of the reduction kernels (0 = any P).
__host__ __device__ constexpr int reduce_pt(int P) { return P == 2 || P == 4 || P == 8 ? P : 0; }

// Below this many bytes per rank a gather job is copied byte by byte: each
// rank then spans at most a handful of 16-byte output vectors, the total is
// at most kMaxRanks * 127 bytes, and the vector machinery would cost more
// than it saves.
constexpr uint64_t kGatherSmallBytes = 128;
// Threads per 16-byte output vector in the small-job part of all_gather_many.
constexpr int kSmallSplit = 4;
// At most this many CTAs copy the small jobs of one launch (one table entry each).
constexpr int kMaxSmallCtas = 512;
// split launch: CTAs of its aligned part and of its realigning part, each at most
constexpr int kMaxPartCtas = 1024;
// split launch, warp realigning: CTAs that copy the unaligned jobs' rank-boundary vectors, at most
constexpr int kMaxBoundaryCtas = 4;

// ------------------------------------------------------------- gather ---
enum : uint32_t {
  kJobFlat = 1u,   // out, bytes and every source are 16-byte aligned
  kJobSmall = 2u,  // bytes < kGatherSmallBytes: byte path
};

// One rank-ordered gather: P sources of `bytes` bytes into out[0, P*bytes).
// Its output is covered by the 16-byte-aligned vectors
// [out/16, (out + P*bytes - 1)/16]; `nvec` counts them and `vfirst` is the
// global index of the first one (prefix over the jobs of one launch).
struct GatherJob {
  uint64_t out;
  uint64_t bytes;
  uint64_t vfirst;
  uint64_t nvec;
  uint32_t src0;   // index of rank 0's source pointer in GatherParams::src
  uint32_t flags;
};

template <int MAXJ, int MAXS>
struct GatherParams {
  uint64_t total_vec;   // sum of nvec over the jobs
  uint64_t flat_vec;    // jobs are ordered aligned (kJobFlat) first: their vectors are [0, flat_vec)
  uint64_t small_vec;   // ... then the other jobs of at least kGatherSmallBytes per rank, then the
                        // kJobSmall jobs, whose vectors are [small_vec, total_vec)
  int32_t small_job0;   // index of the first kJobSmall job (njobs if none)
  int32_t small_ctas;   // split launch: the last small_ctas CTAs copy the kJobSmall jobs
  int32_t njobs;
  int32_t P;
  int32_t staged;       // stage aligned copies through shared memory with cp.async
  int32_t flat_ctas;    // split launch: CTAs [0, flat_ctas) copy the aligned jobs
  int32_t prefetch;     // one aligned job: tiles per CTA prefetched into L2 before the PDL wait
  int32_t tile_vec;     // one job, staged (modes 3, 5): vectors per tile (at most BLOCK*V)
  uint32_t small_per;   // split launch: small-job vectors per small-job CTA (a contiguous run)
  int32_t realign_warp; // one unaligned job: realign across the warp's lanes (mode 6), not through a ring
  uint32_t flat_per;    // split launch: tiles per aligned-part CTA (a contiguous run)
  uint32_t real_per;    // split launch: tiles per realigning-part CTA (a contiguous run)
  int32_t bnd_ctas;     // split launch, warp realigning: CTAs after the realigning part that copy
                        // its jobs' rank-boundary vectors
  GatherJob job[MAXJ];
  uint64_t src[MAXS];   // tensor-major: job j's rank r is src[job[j].src0 + r]
  // split launch: small-job CTA c covers jobs small_job0 + small_tab[c] ..
  // small_job0 + small_tab[c + 1] (the jobs of its first and last vector)
  uint16_t small_tab[MAXJ > 1 ? kMaxSmallCtas + 1 : 1];
  // split launch: the job of the first vector of aligned-part CTA c
  // (flat_tab[c]) and of realigning-part CTA c (real_tab[c])
  uint16_t flat_tab[MAXJ > 1 ? kMaxPartCtas : 1];
  uint16_t real_tab[MAXJ > 1 ? kMaxPartCtas : 1];
};

using GatherParams1 = GatherParams<1, kMaxRanks>;
using GatherParamsS = GatherParams<kManySmallTensors, kManySmallSegments>;
using GatherParamsL = GatherParams<kManyMaxTensors, kManyMaxSegments>;

// One 16-byte aligned gather (out, bytes and every source 16-byte aligned)
// copied by the TMA engine: the output is cut into chunks of `chunk` bytes
// (a multiple of 16), CTA c takes chunks c, c + G, ... and moves each through
// one of `stages` shared-memory stages with 1-D bulk copies.
struct BulkParams {
  uint64_t out;
  uint64_t bytes;      // per rank
  uint64_t total;      // P * bytes
  uint64_t chunk;      // bytes per chunk
  uint64_t wait_ns;    // limit of one wait for a stage's loads (global timer)
  int32_t P;
  int32_t stages;      // ring stages per CTA (1..32)
  int32_t prefetch;    // chunks whose sources a CTA prefetches into L2 ahead of its loads
  uint32_t test_flags; // kBulkTestShortTx: a test makes the first stage's wait run out
  uint64_t src[kMaxRanks];
};
enum : uint32_t { kBulkTestShortTx = 1u };
// Device fault bits (sticky until read by dc_check_device).
enum : uint32_t { kFaultBulkWait = 1u, kFaultFusedWait = 2u };

// The staged all-gather protocol (dc_fused.cu): P ranks, each a group of G
// CTAs of one cooperative launch; rank r's bytes are cut into G chunks of
// `chunk` bytes.  The workspace holds uint32 staged[P][kFusedMaxChunks] and
// done[P][kFusedMaxChunks] epoch flags.
constexpr int kFusedBlock = 256;
constexpr int kFusedMaxChunks = 128;
struct FusedParams {
  uint64_t in[kMaxRanks];
  uint64_t staging[kMaxRanks];
  uint64_t out[kMaxRanks];
  uint64_t bytes;      // per rank, a multiple of 16
  uint64_t chunk;      // a multiple of 16; G * chunk >= bytes
  uint64_t wait_ns;    // limit of one wait (global timer)
  uint64_t ws;         // workspace (device address)
  uint64_t absent;     // (tests) bit r: rank r never arrives
  uint32_t epoch;      // nonzero, new for every call since the workspace was cleared
  int32_t P;
  int32_t G;
  int32_t tma;         // 1: the gather step streams the staged chunks through the TMA engine
  int32_t stages;      // ... in a ring of `stages` shared-memory stages
  uint32_t sub;        // ... of `sub` bytes (a multiple of 16)
};
// Dynamic shared memory of a fused launch (the TMA ring and its mbarriers),
// at most kFusedMaxSmem (the kernel has static shared memory as well).
constexpr size_t kFusedMaxSmem = 226 * 1024;
__host__ __device__ constexpr size_t fused_smem_bytes(int tma, int stages, uint32_t sub) {
  return tma ? static_cast<size_t>(stages) * (static_cast<size_t>(sub) + 8) : 0;
}
__host__ __device__ constexpr size_t fused_workspace_bytes(int P) {
  return static_cast<size_t>(P) * kFusedMaxChunks * 2 * sizeof(uint32_t);
}
cudaError_t launch_fused_gather(const FusedParams& p, cudaStream_t s);
int fused_ctas_per_sm(size_t smem);
// The allocation-free form (dc_fused_all_gather_static): the flags and the
// staging buffers live in a static device array of this many staging bytes
// (rank r's buffer at r * fused_static_stride(bytes)) after the flags of
// kMaxRanks ranks.  launch_fused_gather_static fills p.ws, p.staging and
// p.epoch from it, clears the flags on `s` and launches.
constexpr size_t kFusedStaticStagingBytes = 16u << 20;
__host__ __device__ constexpr uint64_t fused_static_stride(uint64_t bytes) { return (bytes + 255) / 256 * 256; }
cudaError_t launch_fused_gather_static(FusedParams p, cudaStream_t s);
// Reads and clears the first fault of the fused kernel on the current device
// (synchronous): info[0] fault bits, [1] phase << 24 | rank << 12 | peer,
// [2] chunk, [3] epoch.
cudaError_t take_fused_faults(uint32_t* info);

// ---------------------------------------------------------- reduction ---
enum : int { kBF16 = 0, kF16 = 1, kF32 = 2 };              // element types
enum : int { kOrderLinear = 0, kOrderTree = 1 };           // summation orders
enum : uint32_t {
  kJobVec = 1u,      // 16-byte units: every output has the same address mod 16 ...
  kJobRealign = 2u,  // ... and the inputs do not share it: their units are realigned
};

// Batched reductions: at most kManyMaxReduceJobs jobs and kManyMaxReducePtrs
// pointers (inputs and outputs) per launch.
constexpr int kManyMaxReduceJobs = 256;
constexpr int kManyMaxReducePtrs = 1024;

// One fixed-order reduction over `count` elements of one tensor: element i
// reads input q at element in_off + i (input q's pointer is ptr[in0 + q],
// q < P) and writes output m at element i (pointer ptr[out0 + m],
// m < nout).  Work units: an optional scalar head (elements before the
// outputs' first 16-byte boundary), 16-byte vectors, and an optional scalar
// tail; for a job without kJobVec every unit is one element.
struct ReduceJob {
  uint64_t in_off;
  uint64_t count;
  uint64_t ufirst;
  uint64_t nunits;
  uint16_t in0;
  uint16_t out0;
  uint16_t nout;
  uint8_t head;
  uint8_t flags;
};

template <int MAXJ, int MAXPTR>
struct ReduceParams {
  uint64_t total_units;
  int32_t njobs;
  int32_t P;
  int32_t prefetch;     // tiles per CTA whose inputs are prefetched into L2 before the PDL wait
  int32_t tile_units;   // multi-CTA kernel: units per tile (kReduceBlock*unroll, fewer for small launches)
  int32_t staged;       // one realigning all_reduce job through shared memory (dc_reduce_realign_kernel)
  int32_t pad;
  uint64_t ptr[MAXPTR];
  ReduceJob job[MAXJ];
};

using ReduceParams1 = ReduceParams<1, 2 * kMaxRanks>;                        // one all_reduce
using ReduceParamsS = ReduceParams<kMaxRanks, 4 * kMaxRanks>;                // reduce_scatter, small batches
using ReduceParamsL = ReduceParams<kManyMaxReduceJobs, kManyMaxReducePtrs>;  // large batches

// ------------------------------------------------- launch entry points ---
// Each returns the error of the launch itself.  pdl: launch with
// programmatic stream serialization (the kernel may start while the previous
// kernel of the stream drains; it waits for it before touching memory).
cudaError_t launch_gather(const GatherParams1& p, int grid, bool single, bool pdl, cudaStream_t s);
cudaError_t launch_gather(const GatherParamsS& p, int grid, bool single, bool pdl, cudaStream_t s);
cudaError_t launch_gather(const GatherParamsL& p, int grid, bool single, bool pdl, cudaStream_t s);
#define DC_DECLARE_REDUCE(NAME)                                                                  \
  cudaError_t launch_reduce_##NAME(const ReduceParams1& p, int order, int grid, bool single,     \
                                   bool pdl, cudaStream_t s);                                    \
  cudaError_t launch_reduce_##NAME(const ReduceParamsS& p, int order, int grid, bool single,     \
                                   bool pdl, cudaStream_t s);                                    \
  cudaError_t launch_reduce_##NAME(const ReduceParamsL& p, int order, int grid, bool single,     \
                                   bool pdl, cudaStream_t s);                                    \
  int reduce_ctas_per_sm_##NAME(int variant, int order, int P);
DC_DECLARE_REDUCE(bf16)
DC_DECLARE_REDUCE(f16)
DC_DECLARE_REDUCE(f32)
#undef DC_DECLARE_REDUCE

template <class Params>
cudaError_t launch_reduce(const Params& p, int dtype, int order, int grid, bool single, bool pdl,
                          cudaStream_t s) {
  switch (dtype) {
    case kF16: return launch_reduce_f16(p, order, grid, single, pdl, s);
    case kF32: return launch_reduce_f32(p, order, grid, single, pdl, s);
    default: return launch_reduce_bf16(p, order, grid, single, pdl, s);
  }
}

// The TMA-engine gather (dc_bulk.cu): `grid` CTAs, each with `stages` *
// `chunk` bytes of dynamic shared memory (plus its mbarriers).
cudaError_t launch_gather_bulk(const BulkParams& p, int grid, bool pdl, cudaStream_t s);
size_t bulk_smem_bytes(uint64_t chunk, int stages);
constexpr size_t kBulkMaxSmem = 227 * 1024;  // dynamic shared memory one bulk CTA may ask for
// Reads and clears the fault bits that the kernels of dc_bulk.cu recorded on
// the current device (synchronous).
cudaError_t take_bulk_faults(uint32_t* bits);

// Bounds-check records of the checked build (-DDC_DEBUG_BOUNDS), one per
// kernel file; each reads and clears its file's record (synchronous), or
// returns an empty one in the normal build.  bounds_file names the file of
// reader i (i < kBoundsReaders).
struct BoundsFault;
constexpr int kBoundsReaders = 6;
cudaError_t take_bounds_gather(BoundsFault* f);
cudaError_t take_bounds_bulk(BoundsFault* f);
cudaError_t take_bounds_fused(BoundsFault* f);
cudaError_t take_bounds_reduce_bf16(BoundsFault* f);
cudaError_t take_bounds_reduce_f16(BoundsFault* f);
cudaError_t take_bounds_reduce_f32(BoundsFault* f);
bool bounds_checked_build();

// One-thread delay of `ns` nanoseconds of the global timer (rank-skew
// calibration); defined in dc_delay.cu.
cudaError_t launch_delay(unsigned long long ns, cudaStream_t s);

// variant: 0 ReduceParams1, 1 ReduceParamsS, 2 ReduceParamsL, 3 the staged
// realigning kernel (ReduceParams1).
inline int reduce_ctas_per_sm(int dtype, int variant, int order, int P) {
  switch (dtype) {
    case kF16: return reduce_ctas_per_sm_f16(variant, order, P);
    case kF32: return reduce_ctas_per_sm_f32(variant, order, P);
    default: return reduce_ctas_per_sm_bf16(variant, order, P);
  }
}

// cudaLaunchKernelEx with an optional programmatic-serialization attribute.
template <typename Kernel, typename Params>
cudaError_t launch_ex(Kernel kernel, int grid, int block, bool pdl, cudaStream_t s, const Params& p,
                      size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Resident CTAs per SM of the multi-CTA kernels (occupancy API, per device).
int gather_ctas_per_sm(int which, int mode);  // which: 0 one job, 1 small many, 2 large many
// Kernel mode a launch will use: 0 general, 1 aligned jobs, 2 one aligned job,
// 3 one aligned job staged through shared memory, 4 (kGatherModeSplit) several
// jobs, the aligned ones staged by the first flat_ctas CTAs, 5 one unaligned
// job staged through shared memory, 6 (kGatherModeWarpRealign) one unaligned
// job realigned across the lanes of a warp.
constexpr int kGatherModeSplit = 4;
constexpr int kGatherModeWarpRealign = 6;
constexpr int kGatherModes = 7;
int gather_mode_of(const GatherParams1& p);
int gather_mode_of(const GatherParamsS& p);
int gather_mode_of(const GatherParamsL& p);

}  // namespace dc
