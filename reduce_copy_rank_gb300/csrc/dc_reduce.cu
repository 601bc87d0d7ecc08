// dc_reduce.cu -- the deterministic BF16 all_reduce / reduce_scatter fold.
//
// "perf(cuda): vectorize the deterministic all-gather copy and right-size its
// single-block path" (RL-Kernel PR 491) names the deterministic all_reduce
// and reduce_scatter (sections "What" and "Not in this PR": their single-block
// paths grow linearly with size, 523 us at 256 KiB vs 70 us at 512 KiB on
// eight B200s) and, in the author's replies, the reduce_scatter shape: the
// input is world x output, as in torch's reduce_scatter_tensor.  The page
// never prints the arithmetic.  The reading implemented here, which makes the
// result independent of scheduling: for every element, start from rank 0's
// value widened to binary32, add ranks 1..P-1 one at a time in binary32
// (round to nearest even), and round the total once to BF16 (round to nearest
// even).  No reassociation, no tree, no cross-thread combine: each thread
// folds its own elements, so the bits do not depend on grid, block or vector
// width.  Subnormals are kept (built without flush-to-zero).
//
// Layout of the work: a job is one contiguous element range with one input
// offset (all_reduce: one job writing P outputs; reduce_scatter: P jobs, job
// r reading elements [r*C, (r+1)*C) of every input and writing output r).
// When every pointer of a job has the same address mod 16, the job is a
// scalar head up to the first 16-byte boundary, a body of 8-element groups
// (one 16-byte load per rank and one 16-byte store per output, P loads in
// flight per group) and a scalar tail.  Otherwise every element is folded
// with 2-byte accesses.  CTAs take tiles of units round robin and find a
// tile's job by walking the job table forward; there is no per-element
// division.
#include "dc_device.cuh"
#include "dc_internal.h"

namespace dc {
namespace {

template <int MAXJ>
__device__ __forceinline__ float load_bf16(const ReduceParams<MAXJ>& p, int q, uint64_t elem) {
  const uint16_t h = *reinterpret_cast<const uint16_t*>(p.in[q] + 2 * elem);
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Elements [e0, e1) of job J, one at a time.
template <int MAXJ>
__device__ __forceinline__ void fold_scalar(const ReduceParams<MAXJ>& p, const ReduceJob& J,
                                            uint64_t e0, uint64_t e1, uint64_t step) {
  for (uint64_t i = e0; i < e1; i += step) {
    const uint64_t elem = J.in_off + i;
    float acc = load_bf16(p, 0, elem);
    for (int q = 1; q < p.P; ++q) acc = __fadd_rn(acc, load_bf16(p, q, elem));
    const uint16_t y = f32_to_bf16_rn(acc);
    for (uint32_t m = 0; m < J.nout; ++m)
      *reinterpret_cast<uint16_t*>(p.out[J.out0 + m] + 2 * i) = y;
  }
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&a)[8]) {
  a[0] = bf16lo_to_f32(v.x); a[1] = bf16hi_to_f32(v.x);
  a[2] = bf16lo_to_f32(v.y); a[3] = bf16hi_to_f32(v.y);
  a[4] = bf16lo_to_f32(v.z); a[5] = bf16hi_to_f32(v.z);
  a[6] = bf16lo_to_f32(v.w); a[7] = bf16hi_to_f32(v.w);
}

__device__ __forceinline__ void add8(float (&a)[8], const uint4& v) {
  a[0] = __fadd_rn(a[0], bf16lo_to_f32(v.x)); a[1] = __fadd_rn(a[1], bf16hi_to_f32(v.x));
  a[2] = __fadd_rn(a[2], bf16lo_to_f32(v.y)); a[3] = __fadd_rn(a[3], bf16hi_to_f32(v.y));
  a[4] = __fadd_rn(a[4], bf16lo_to_f32(v.z)); a[5] = __fadd_rn(a[5], bf16hi_to_f32(v.z));
  a[6] = __fadd_rn(a[6], bf16lo_to_f32(v.w)); a[7] = __fadd_rn(a[7], bf16hi_to_f32(v.w));
}

__device__ __forceinline__ uint4 pack8(const float (&a)[8]) {
  uint4 r;
  r.x = pack_bf16x2_rn(a[0], a[1]);
  r.y = pack_bf16x2_rn(a[2], a[3]);
  r.z = pack_bf16x2_rn(a[4], a[5]);
  r.w = pack_bf16x2_rn(a[6], a[7]);
  return r;
}

// Loads of one 8-element group at input element `elem` (16-byte aligned in
// every input) and its fold.  PT > 0: P known at compile time, and the caller
// issues the loads of all its groups before the first add.  PT == 0: ranks
// in batches of 8 loads.
template <int PT, int MAXJ>
__device__ __forceinline__ void load_group(const ReduceParams<MAXJ>& p, uint64_t elem,
                                           uint4 (&v)[PT > 0 ? PT : 1]) {
#pragma unroll
  for (int q = 0; q < (PT > 0 ? PT : 1); ++q)
    v[q] = ld_stream(reinterpret_cast<const uint4*>(p.in[q] + 2 * elem));
}

template <int PT, int MAXJ>
__device__ __forceinline__ void fold_loaded(const ReduceParams<MAXJ>& p, uint64_t elem,
                                            const uint4 (&v)[PT > 0 ? PT : 1], float (&acc)[8]) {
  unpack8(v[0], acc);
  if constexpr (PT > 0) {
#pragma unroll
    for (int q = 1; q < PT; ++q) add8(acc, v[q]);
  } else {
    for (int q0 = 1; q0 < p.P; q0 += 8) {
      uint4 w[8];
      const int nb = min(8, p.P - q0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < nb) w[k] = ld_stream(reinterpret_cast<const uint4*>(p.in[q0 + k] + 2 * elem));
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < nb) add8(acc, w[k]);
    }
  }
}

template <int BLOCK, int UNROLL, int PT, int MAXJ>
__device__ __forceinline__ void reduce_job_vec(const ReduceParams<MAXJ>& p, const ReduceJob& J,
                                               uint64_t a, uint64_t b) {
  const uint64_t hu = J.head ? 1 : 0;
  const uint64_t nbody = (J.count - J.head) >> 3;
  const uint64_t tail_unit = hu + nbody;
  const bool has_tail = ((J.count - J.head) & 7u) != 0;
  if (hu && a == 0 && threadIdx.x == 0) fold_scalar(p, J, 0, J.head, 1);
  if (has_tail && a <= tail_unit && tail_unit < b && threadIdx.x == BLOCK - 1)
    fold_scalar(p, J, J.head + 8 * nbody, J.count, 1);
  const uint64_t ba = max(a, hu), bb = min(b, tail_unit);
  for (uint64_t u0 = ba + threadIdx.x; u0 < bb; u0 += BLOCK * UNROLL) {
    uint4 v[UNROLL][PT > 0 ? PT : 1];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const uint64_t u = u0 + k * BLOCK;
      if (u < bb) load_group<PT>(p, J.in_off + J.head + 8 * (u - hu), v[k]);
    }
    float acc[UNROLL][8];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const uint64_t u = u0 + k * BLOCK;
      if (u < bb) fold_loaded<PT>(p, J.in_off + J.head + 8 * (u - hu), v[k], acc[k]);
    }
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const uint64_t u = u0 + k * BLOCK;
      if (u < bb) {
        const uint4 y = pack8(acc[k]);
        const uint64_t byte_off = 2 * (J.head + 8 * (u - hu));
        for (uint32_t m = 0; m < J.nout; ++m)
          st16(reinterpret_cast<uint4*>(p.out[J.out0 + m] + byte_off), y);
      }
    }
  }
}

// Tile t covers global units [t*TILE, (t+1)*TILE), TILE = BLOCK*UNROLL; a
// CTA takes tiles first, first + step, ...  so that all CTAs sweep the
// buffers together (neighbouring CTAs read neighbouring addresses), which
// keeps DRAM rows and TLB entries shared between them.
template <int BLOCK, int UNROLL, int PT, int MAXJ>
__device__ __forceinline__ void reduce_tiles(const ReduceParams<MAXJ>& p, uint64_t first,
                                             uint64_t step) {
  constexpr uint64_t kTile = static_cast<uint64_t>(BLOCK) * UNROLL;
  const uint64_t ntiles = (p.total_units + kTile - 1) / kTile;
  int j = 0;
  for (uint64_t t = first; t < ntiles; t += step) {
    const uint64_t g0 = t * kTile, g1 = min(g0 + kTile, p.total_units);
    while (j + 1 < p.njobs && p.job[j].ufirst + p.job[j].nunits <= g0) ++j;
    for (int jj = j; jj < p.njobs && p.job[jj].ufirst < g1; ++jj) {
      const ReduceJob& J = p.job[jj];
      const uint64_t a = max(g0, J.ufirst) - J.ufirst;
      const uint64_t b = min(g1, J.ufirst + J.nunits) - J.ufirst;
      if (a >= b) continue;
      if (J.flags & kJobVec)
        reduce_job_vec<BLOCK, UNROLL, PT>(p, J, a, b);
      else
        fold_scalar(p, J, a + threadIdx.x, b, BLOCK);
    }
  }
}

template <int MAXJ, int PT>
__global__ void __launch_bounds__(kReduceBlock)
    dc_reduce_kernel(const __grid_constant__ ReduceParams<MAXJ> p) {
  pdl_enter();
  reduce_tiles<kReduceBlock, kReduceUnroll, PT>(p, blockIdx.x, gridDim.x);
}

template <int MAXJ, int PT>
__global__ void __launch_bounds__(kReduceSingleBlock)
    dc_reduce_single_kernel(const __grid_constant__ ReduceParams<MAXJ> p) {
  pdl_enter();
  reduce_tiles<kReduceSingleBlock, kReduceUnroll, PT>(p, 0, 1);
}

template <int MAXJ, int PT>
cudaError_t launch_pt(const ReduceParams<MAXJ>& p, int grid, bool single, bool pdl, cudaStream_t s) {
  if (single) return launch_ex(dc_reduce_single_kernel<MAXJ, PT>, 1, kReduceSingleBlock, pdl, s, p);
  return launch_ex(dc_reduce_kernel<MAXJ, PT>, grid, kReduceBlock, pdl, s, p);
}

template <int MAXJ>
cudaError_t launch_impl(const ReduceParams<MAXJ>& p, int grid, bool single, bool pdl,
                        cudaStream_t s) {
  switch (p.P) {
    case 8: return launch_pt<MAXJ, 8>(p, grid, single, pdl, s);
    case 4: return launch_pt<MAXJ, 4>(p, grid, single, pdl, s);
    case 2: return launch_pt<MAXJ, 2>(p, grid, single, pdl, s);
    default: return launch_pt<MAXJ, 0>(p, grid, single, pdl, s);
  }
}

template <int MAXJ, int PT>
int occupancy_pt() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dc_reduce_kernel<MAXJ, PT>, kReduceBlock,
                                                    0) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return n > 0 ? n : 1;
}

template <int MAXJ>
int occupancy_impl(int P) {
  switch (P) {
    case 8: return occupancy_pt<MAXJ, 8>();
    case 4: return occupancy_pt<MAXJ, 4>();
    case 2: return occupancy_pt<MAXJ, 2>();
    default: return occupancy_pt<MAXJ, 0>();
  }
}

}  // namespace

cudaError_t launch_reduce(const ReduceParams1& p, int grid, bool single, bool pdl, cudaStream_t s) {
  return launch_impl(p, grid, single, pdl, s);
}
cudaError_t launch_reduce(const ReduceParamsP& p, int grid, bool single, bool pdl, cudaStream_t s) {
  return launch_impl(p, grid, single, pdl, s);
}

int reduce_ctas_per_sm(int P, bool scatter) {
  return scatter ? occupancy_impl<kMaxRanks>(P) : occupancy_impl<1>(P);
}

}  // namespace dc
