// dc_reduce.cuh -- the deterministic fixed-order reductions (all_reduce,
// reduce_scatter and their batched forms) for BF16, FP16 and FP32, in the
// linear or the tree summation order.  Included by one .cu file per element
// type, which instantiates the kernels for that type.
//
// "perf(cuda): vectorize the deterministic all-gather copy and right-size its
// single-block path" (RL-Kernel PR 491) names the deterministic all_reduce
// and reduce_scatter (sections "What" and "Not in this PR": their single-block
// paths grow linearly with size), their batched form (reduce_scatter_many,
// whose outs= argument upstream rejected), the reduce_scatter shape (author's
// reply: input = world x output) and a backend called "cuda_ipc_fixed_tree".
// The page never prints the arithmetic.  The reading implemented here: every
// element of every rank is widened exactly to binary32; the P values of one
// element are added in a fixed order, one binary32 add (round to nearest
// even) at a time:
//   linear: ((x0 + x1) + x2) + ... + x_{P-1};
//   tree:   fold(x[lo..hi)) = fold(x[lo..lo+m)) + fold(x[lo+m..hi)), m the
//           largest power of two below hi - lo (pairs of neighbouring ranks,
//           then pairs of pairs; a trailing odd group is added last);
// and the binary32 total is rounded once to the element type (round to
// nearest even; FP32 totals are stored as they are).  No reassociation and no
// cross-thread combine: each thread folds its own elements, so the bits do
// not depend on grid, block or vector width.  Subnormals are kept.
//
// Work: a job is one contiguous element range of one tensor with one input
// offset (all_reduce: one job per tensor, writing P outputs; reduce_scatter:
// one job per tensor and rank r, reading elements [r*C, (r+1)*C) of the
// tensor's inputs and writing output r).  When the outputs of a job share
// one address mod 16, the job is a scalar head up to the outputs' first
// 16-byte boundary, a body of 16-byte units (one store per output) and a
// scalar tail; an input at the outputs' offset is read with one 16-byte load
// per unit, an input at another offset as the two aligned blocks around the
// unit, funnel-shifted (in registers, or for an all_reduce of one tensor with
// P = 2, 4, 8 through shared memory: reduce_realign_staged).  When the
// outputs disagree mod 16 the job is folded element by element.  Units are
// taken in tiles round robin by the CTAs; a one-tensor all_reduce's tiles are
// sized by the planner so that every SM gets the same share.
#pragma once

#include <atomic>

#include "dc_device.cuh"
#include "dc_internal.h"

namespace dc {
namespace red {

// ------------------------------------------------------- element types ---
template <int DT>
struct Elem;

template <>
struct Elem<kBF16> {
  static constexpr int kSize = 2, kPerVec = 8;
  using Raw = uint16_t;
  __device__ static __forceinline__ float widen1(Raw h) { return __uint_as_float(uint32_t{h} << 16); }
  __device__ static __forceinline__ Raw narrow1(float x) { return f32_to_bf16_rn(x); }
  __device__ static __forceinline__ void widen(const uint4& v, float (&a)[kPerVec]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a[2 * i] = bf16lo_to_f32(w[i]);
      a[2 * i + 1] = bf16hi_to_f32(w[i]);
    }
  }
  __device__ static __forceinline__ uint4 narrow(const float (&a)[kPerVec]) {
    return make_uint4(pack_bf16x2_rn(a[0], a[1]), pack_bf16x2_rn(a[2], a[3]),
                      pack_bf16x2_rn(a[4], a[5]), pack_bf16x2_rn(a[6], a[7]));
  }
};

template <>
struct Elem<kF16> {
  static constexpr int kSize = 2, kPerVec = 8;
  using Raw = uint16_t;
  __device__ static __forceinline__ float widen1(Raw h) { return f16_to_f32(h); }
  __device__ static __forceinline__ Raw narrow1(float x) { return f32_to_f16_rn(x); }
  __device__ static __forceinline__ void widen(const uint4& v, float (&a)[kPerVec]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a[2 * i] = f16_to_f32(static_cast<uint16_t>(w[i] & 0xFFFFu));
      a[2 * i + 1] = f16_to_f32(static_cast<uint16_t>(w[i] >> 16));
    }
  }
  __device__ static __forceinline__ uint4 narrow(const float (&a)[kPerVec]) {
    return make_uint4(pack_f16x2_rn(a[0], a[1]), pack_f16x2_rn(a[2], a[3]),
                      pack_f16x2_rn(a[4], a[5]), pack_f16x2_rn(a[6], a[7]));
  }
};

template <>
struct Elem<kF32> {
  static constexpr int kSize = 4, kPerVec = 4;
  using Raw = uint32_t;
  __device__ static __forceinline__ float widen1(Raw u) { return __uint_as_float(u); }
  __device__ static __forceinline__ Raw narrow1(float x) { return __float_as_uint(x); }
  __device__ static __forceinline__ void widen(const uint4& v, float (&a)[kPerVec]) {
    a[0] = __uint_as_float(v.x);
    a[1] = __uint_as_float(v.y);
    a[2] = __uint_as_float(v.z);
    a[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ uint4 narrow(const float (&a)[kPerVec]) {
    return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                      __float_as_uint(a[3]));
  }
};

// -------------------------------------------------------------- folds ---
template <int E>
__device__ __forceinline__ void add_into(float (&acc)[E], const float (&x)[E]) {  // acc = acc + x
#pragma unroll
  for (int i = 0; i < E; ++i) acc[i] = __fadd_rn(acc[i], x[i]);
}

template <int E>
__device__ __forceinline__ void add_left(const float (&left)[E], float (&acc)[E]) {  // acc = left + acc
#pragma unroll
  for (int i = 0; i < E; ++i) acc[i] = __fadd_rn(left[i], acc[i]);
}

// Tree fold with a stack of partial sums: rank q enters as a leaf of level 0;
// while the top of the stack has the same level, the two merge (older on the
// left) into one of the next level; at the end the stack is folded from the
// top down, each entry added on the left.  This builds exactly
// fold(lo..hi) = fold(lo..lo+m) + fold(lo+m..hi) with m the largest power of
// two below hi - lo.
template <int E>
struct TreeStack {
  static constexpr int kDepth = 7;  // P <= 64
  float s[kDepth][E];
  int level[kDepth];
  int n = 0;
  __device__ __forceinline__ void push(float (&x)[E]) {
    int l = 0;
    while (n > 0 && level[n - 1] == l) {
      add_left(s[n - 1], x);  // x = s[top] + x
      --n;
      ++l;
    }
#pragma unroll
    for (int i = 0; i < E; ++i) s[n][i] = x[i];
    level[n] = l;
    ++n;
  }
  __device__ __forceinline__ void finish(float (&acc)[E]) {
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = s[n - 1][i];
    for (int k = n - 2; k >= 0; --k) add_left(s[k], acc);
  }
};

// ------------------------------------------------------------- params ---
template <int MAXJ, int MAXPTR>
__device__ __forceinline__ const uint8_t* in_ptr(const ReduceParams<MAXJ, MAXPTR>& p,
                                                 const ReduceJob& J, int q) {
  return reinterpret_cast<const uint8_t*>(p.ptr[J.in0 + q]);
}
template <int MAXJ, int MAXPTR>
__device__ __forceinline__ uint8_t* out_ptr(const ReduceParams<MAXJ, MAXPTR>& p, const ReduceJob& J,
                                            int m) {
  return reinterpret_cast<uint8_t*>(p.ptr[J.out0 + m]);
}

// Bounds checks of the checked build (in_bounds): job J may read of input q
// the 16-byte-block hull of its element range [in_q + in_off*s, in_q +
// (in_off + count)*s), and write of output m exactly [out_m, out_m +
// count*s).  Sites, for the fault record: kSiteRed* below.
enum : uint32_t {
  kSiteRedScalar = 200, kSiteRedVec = 201, kSiteRedStaged = 202, kSiteRedPrefetch = 203,
};
template <int DT, int MAXJ, int MAXPTR>
__device__ __forceinline__ bool input_ok(const ReduceParams<MAXJ, MAXPTR>& p, const ReduceJob& J, int q,
                                         const void* a, uint64_t len, uint32_t site) {
  const uint64_t base = reinterpret_cast<uint64_t>(in_ptr(p, J, q)) + J.in_off * Elem<DT>::kSize;
  return in_bounds(a, len, hull_lo(base), hull_hi(base, J.count * Elem<DT>::kSize), site);
}
template <int DT, int MAXJ, int MAXPTR>
__device__ __forceinline__ bool output_ok(const ReduceParams<MAXJ, MAXPTR>& p, const ReduceJob& J, int m,
                                          const void* a, uint64_t len, uint32_t site) {
  const uint64_t base = reinterpret_cast<uint64_t>(out_ptr(p, J, m));
  return in_bounds(a, len, base, base + J.count * Elem<DT>::kSize, site);
}

// The 16 input bytes of rank q at `a`.  A job whose inputs all share the
// outputs' address mod 16 loads them with one aligned load; a realigning job
// (inputs at other offsets) loads the aligned block holding `a` and, if `a`
// is not 16-byte aligned, the next one, and funnel-shifts them.  Both blocks
// hold bytes of [a, a + 16), so they lie in the input buffer; a thread's
// second block is its neighbour's first (coherent, L1-allocating load: a job
// may run in place).
template <bool REALIGN, int DT, int MAXJ, int MAXPTR>
__device__ __forceinline__ uint4 ld_input(const ReduceParams<MAXJ, MAXPTR>& p, const ReduceJob& J, int q,
                                          const uint8_t* a) {
  uint4 lo = make_uint4(0, 0, 0, 0);
  if constexpr (!REALIGN) {
    const uint4* v = reinterpret_cast<const uint4*>(a);
    if (input_ok<DT>(p, J, q, v, 16, kSiteRedVec)) lo = ld_stream(v);
    return lo;
  } else {
    const uint32_t s = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(a) & 15u);
    const uint4* blk = reinterpret_cast<const uint4*>(a - s);
    if (input_ok<DT>(p, J, q, blk, 16, kSiteRedVec)) lo = ld_cached(blk);
    uint4 hi = lo;
    if (s && input_ok<DT>(p, J, q, blk + 1, 16, kSiteRedVec)) hi = ld_cached(blk + 1);
    return realign16(lo, hi, s);
  }
}

// One element of rank q at `a` (checked build: inside the job's range).
template <int DT, int MAXJ, int MAXPTR>
__device__ __forceinline__ float ld_element(const ReduceParams<MAXJ, MAXPTR>& p, const ReduceJob& J, int q,
                                            const uint8_t* a) {
  using Raw = typename Elem<DT>::Raw;
  if (!input_ok<DT>(p, J, q, a, sizeof(Raw), kSiteRedScalar)) return 0.0f;
  return Elem<DT>::widen1(*reinterpret_cast<const Raw*>(a));
}

// Elements [e0, e1) (step `step`) of job J, one at a time.
template <int DT, int ORDER, int MAXJ, int MAXPTR>
__device__ __forceinline__ void fold_scalar(const ReduceParams<MAXJ, MAXPTR>& p, const ReduceJob& J,
                                            uint64_t e0, uint64_t e1, uint64_t step) {
  using T = Elem<DT>;
  using Raw = typename T::Raw;
  for (uint64_t i = e0; i < e1; i += step) {
    const uint64_t off = (J.in_off + i) * T::kSize;
    float acc[1];
    if (ORDER == kOrderTree) {
      TreeStack<1> st;
      for (int q = 0; q < p.P; ++q) {
        float x[1] = {ld_element<DT>(p, J, q, in_ptr(p, J, q) + off)};
        st.push(x);
      }
      st.finish(acc);
    } else {
      acc[0] = ld_element<DT>(p, J, 0, in_ptr(p, J, 0) + off);
      for (int q = 1; q < p.P; ++q) acc[0] = __fadd_rn(acc[0], ld_element<DT>(p, J, q, in_ptr(p, J, q) + off));
    }
    const Raw y = T::narrow1(acc[0]);
    for (uint32_t m = 0; m < J.nout; ++m) {
      Raw* d = reinterpret_cast<Raw*>(out_ptr(p, J, m) + i * T::kSize);
      if (output_ok<DT>(p, J, m, d, sizeof(Raw), kSiteRedScalar)) *d = y;
    }
  }
}

// The fold of one 16-byte vector of every rank at byte offset `off` of each
// input.  PT > 0: P = PT known at compile time, all loads issued first by the
// caller (`v`).  PT == 0: ranks in batches of 8 loads.
template <int DT, int ORDER, int PT, bool REALIGN, int MAXJ, int MAXPTR>
__device__ __forceinline__ void fold_vector(const ReduceParams<MAXJ, MAXPTR>& p, const ReduceJob& J,
                                            uint64_t off, const uint4 (&v)[PT > 0 ? PT : 1],
                                            float (&acc)[Elem<DT>::kPerVec]) {
  using T = Elem<DT>;
  constexpr int E = T::kPerVec;
  if constexpr (PT > 0) {
    float x[PT][E];
#pragma unroll
    for (int q = 0; q < PT; ++q) T::widen(v[q], x[q]);
    if constexpr (ORDER == kOrderTree) {
      // levels of a complete binary tree over PT = 2^k leaves, left + right
#pragma unroll
      for (int width = 1; width < PT; width *= 2)
#pragma unroll
        for (int q = 0; q + width < PT; q += 2 * width) add_into(x[q], x[q + width]);
#pragma unroll
      for (int i = 0; i < E; ++i) acc[i] = x[0][i];
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) acc[i] = x[0][i];
#pragma unroll
      for (int q = 1; q < PT; ++q) add_into(acc, x[q]);
    }
  } else {
    TreeStack<E> st;
    for (int q0 = 0; q0 < p.P; q0 += 8) {
      uint4 w[8];
      const int nb = min(8, p.P - q0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < nb) w[k] = ld_input<REALIGN, DT>(p, J, q0 + k, in_ptr(p, J, q0 + k) + off);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < nb) {
          float x[E];
          T::widen(w[k], x);
          if constexpr (ORDER == kOrderTree) {
            st.push(x);
          } else if (q0 + k == 0) {
#pragma unroll
            for (int i = 0; i < E; ++i) acc[i] = x[i];
          } else {
            add_into(acc, x);
          }
        }
      }
    }
    if constexpr (ORDER == kOrderTree) st.finish(acc);
  }
}

template <int DT, int ORDER, int BLOCK, int UNROLL, int PT, bool REALIGN, int MAXJ, int MAXPTR>
__device__ __forceinline__ void reduce_job_vec(const ReduceParams<MAXJ, MAXPTR>& p,
                                               const ReduceJob& J, uint64_t a, uint64_t b) {
  using T = Elem<DT>;
  constexpr int E = T::kPerVec;
  const uint64_t hu = J.head ? 1 : 0;
  const uint64_t nbody = (J.count - J.head) / E;
  const uint64_t tail_unit = hu + nbody;
  const bool has_tail = ((J.count - J.head) % E) != 0;
  if (hu && a == 0 && threadIdx.x == 0) fold_scalar<DT, ORDER>(p, J, 0, J.head, 1);
  if (has_tail && a <= tail_unit && tail_unit < b && threadIdx.x == BLOCK - 1)
    fold_scalar<DT, ORDER>(p, J, J.head + E * nbody, J.count, 1);
  const uint64_t ba = max(a, hu), bb = min(b, tail_unit);
  for (uint64_t u0 = ba + threadIdx.x; u0 < bb; u0 += BLOCK * UNROLL) {
    uint4 v[UNROLL][PT > 0 ? PT : 1];
    if constexpr (PT > 0) {
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        const uint64_t u = u0 + k * BLOCK;
        if (u < bb) {
          const uint64_t off = (J.in_off + J.head + E * (u - hu)) * T::kSize;
#pragma unroll
          for (int q = 0; q < PT; ++q)
            v[k][q] = ld_input<REALIGN, DT>(p, J, q, in_ptr(p, J, q) + off);
        }
      }
    }
    // group by group: one accumulator live at a time, however many groups
    // are in flight
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      const uint64_t u = u0 + k * BLOCK;
      if (u < bb) {
        float acc[E];
        fold_vector<DT, ORDER, PT, REALIGN>(p, J, (J.in_off + J.head + E * (u - hu)) * T::kSize, v[k],
                                            acc);
        const uint4 y = T::narrow(acc);
        const uint64_t byte_off = (J.head + E * (u - hu)) * T::kSize;
        for (uint32_t m = 0; m < J.nout; ++m) {
          uint4* d = reinterpret_cast<uint4*>(out_ptr(p, J, m) + byte_off);
          if (output_ok<DT>(p, J, m, d, 16, kSiteRedVec)) st16(d, y);
        }
      }
    }
  }
}

// Tile t covers global units [t*tile, (t+1)*tile) (tile = BLOCK*UNROLL, or
// fewer units so that a small launch reaches every SM); a CTA takes tiles
// first, first + step, ... so that all CTAs sweep the buffers together.  A
// tile's job is found by walking the job table forward.
template <int DT, int ORDER, int BLOCK, int UNROLL, int PT, int MAXJ, int MAXPTR>
__device__ __forceinline__ void reduce_tiles(const ReduceParams<MAXJ, MAXPTR>& p, uint64_t tile,
                                             uint64_t first, uint64_t step) {
  const uint64_t ntiles = (p.total_units + tile - 1) / tile;
  int j = 0;
  for (uint64_t t = first; t < ntiles; t += step) {
    const uint64_t g0 = t * tile, g1 = min(g0 + tile, p.total_units);
    while (j + 1 < p.njobs && p.job[j].ufirst + p.job[j].nunits <= g0) ++j;
    for (int jj = j; jj < p.njobs && p.job[jj].ufirst < g1; ++jj) {
      const ReduceJob& J = p.job[jj];
      const uint64_t a = max(g0, J.ufirst) - J.ufirst;
      const uint64_t b = min(g1, J.ufirst + J.nunits) - J.ufirst;
      if (a >= b) continue;
      if ((J.flags & (kJobVec | kJobRealign)) == kJobVec)
        reduce_job_vec<DT, ORDER, BLOCK, UNROLL, PT, false>(p, J, a, b);
      else if (J.flags & kJobVec)  // realigned inputs: two loads each, half as many groups in flight
        reduce_job_vec<DT, ORDER, BLOCK, (UNROLL > 1 ? UNROLL / 2 : 1), PT, true>(p, J, a, b);
      else
        fold_scalar<DT, ORDER>(p, J, a + threadIdx.x, b, BLOCK);
    }
  }
}

// The 16-byte input vectors of tile t prefetched into L2, thread q < P
// taking rank q (one bulk prefetch per job the tile overlaps; scalar heads
// and tails are left out).  Issued before the PDL wait, so the HBM latency
// of the first tiles overlaps the end of the previous kernel in the stream.
template <int DT, int MAXJ, int MAXPTR>
__device__ __forceinline__ void reduce_prefetch_tile(const ReduceParams<MAXJ, MAXPTR>& p,
                                                     uint64_t tile, uint64_t t) {
  using T = Elem<DT>;
  constexpr int E = T::kPerVec;
  const uint64_t g0 = t * tile;
  if (g0 >= p.total_units || threadIdx.x >= static_cast<unsigned>(p.P)) return;
  const uint64_t g1 = min(g0 + tile, p.total_units);
  for (int jj = 0; jj < p.njobs && p.job[jj].ufirst < g1; ++jj) {
    const ReduceJob& J = p.job[jj];
    if (J.ufirst + J.nunits <= g0 || (J.flags & (kJobVec | kJobRealign)) != kJobVec) continue;
    const uint64_t hu = J.head ? 1 : 0;
    const uint64_t body_end = hu + (J.count - J.head) / E;
    const uint64_t a = max(max(g0, J.ufirst) - J.ufirst, hu);
    const uint64_t b = min(min(g1, J.ufirst + J.nunits) - J.ufirst, body_end);
    if (a >= b) continue;
    const uint8_t* src = in_ptr(p, J, threadIdx.x) + (J.in_off + J.head + E * (a - hu)) * T::kSize;
    if (input_ok<DT>(p, J, threadIdx.x, src, (b - a) * 16, kSiteRedPrefetch))
      prefetch_l2(src, static_cast<uint32_t>((b - a) * 16));
  }
}

// One all_reduce job (one tensor) whose inputs do not all share the outputs'
// address mod 16 (kJobVec | kJobRealign), P = PT known at compile time.  The
// register path loads two 16-byte blocks per realigned input and so keeps
// half as many units in flight; here the input blocks go through shared
// memory instead.  Tile t is body units [t*BLOCK, (t+1)*BLOCK); a CTA takes
// tiles first, first + step, ... through a ring of S stages.  Per stage, rank
// and warp the ring holds 33 blocks: lane l copies (cp.async, L2 only) the
// aligned block holding its unit's first input byte into slot l; a realigned
// rank's unit also needs the next block, which is lane l+1's, so only the
// last active lane of the warp copies it, into slot l+1.  After its own
// copies are in (cp.async.wait_group) a lane synchronises with its warp
// (__syncwarp orders the lanes' shared-memory accesses), reads slots l and
// l+1, funnel-shifts them (realign16) and folds the P vectors exactly as the
// register path does (fold_vector), so the bits are the same; a second
// __syncwarp keeps slot l from being refilled before lane l-1 has read it.
// In place: an output may be exactly its rank's input; that rank then has the
// outputs' offset (no second block), and its unit's block is copied in before
// the same thread writes the unit.  The scalar head and tail (fewer than 16
// bytes each) are folded by threads 0 and BLOCK-1 of the first CTA.
template <int DT, int ORDER, int BLOCK, int PT, int S, int MAXJ, int MAXPTR>
__device__ __forceinline__ void reduce_realign_staged(const ReduceParams<MAXJ, MAXPTR>& p, uint64_t first,
                                                      uint64_t step) {
  using T = Elem<DT>;
  constexpr int E = T::kPerVec;
  constexpr uint32_t kRow = 33;                                   // slots per warp, rank and stage
  constexpr uint32_t kRank = 16u * kRow * (BLOCK / 32);           // bytes per rank and stage
  extern __shared__ uint4 red_stage[];                            // [S][PT][BLOCK/32][kRow]
  const ReduceJob& J = p.job[0];
  const uint64_t nbody = (J.count - J.head) / E;
  const uint64_t ntiles = (nbody + BLOCK - 1) / BLOCK;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(red_stage)) +
                         16u * ((threadIdx.x >> 5) * kRow + lane);
  // input byte address of body unit 0 of rank q (unit b starts 16*b later)
  auto in0 = [&](int q) {
    return reinterpret_cast<uint64_t>(in_ptr(p, J, q)) + (J.in_off + J.head) * T::kSize;
  };
  auto issue = [&](uint32_t slot, uint64_t t) {
    const uint64_t b = t * BLOCK + threadIdx.x;
    if (t < ntiles && b < nbody) {
      const bool last = lane == 31u || b + 1 >= nbody;  // the warp's last active lane
#pragma unroll
      for (int q = 0; q < PT; ++q) {
        const uint64_t a = in0(q) + 16 * b;
        const uint64_t blk = a & ~static_cast<uint64_t>(15);
        const uint32_t dst = sbase + kRank * (slot * PT + q);
        if (input_ok<DT>(p, J, q, reinterpret_cast<const void*>(blk), 16, kSiteRedStaged))
          cp_async16(dst, reinterpret_cast<const void*>(blk));
        if ((a & 15u) && last && input_ok<DT>(p, J, q, reinterpret_cast<const void*>(blk + 16), 16, kSiteRedStaged))
          cp_async16(dst + 16u, reinterpret_cast<const void*>(blk + 16));
      }
    }
    cp_async_commit();
  };
  uint64_t t_issue = first;
#pragma unroll
  for (int i = 0; i < S; ++i) {
    issue(static_cast<uint32_t>(i), t_issue);
    t_issue += step;
  }
  if (first == 0) {  // scalar head and tail, while the ring fills
    const uint64_t tail0 = J.head + static_cast<uint64_t>(E) * nbody;
    if (J.head && threadIdx.x == 0) fold_scalar<DT, ORDER>(p, J, 0, J.head, 1);
    if (tail0 < J.count && threadIdx.x == BLOCK - 1) fold_scalar<DT, ORDER>(p, J, tail0, J.count, 1);
  }
  uint32_t slot = 0;
  for (uint64_t t = first; t < ntiles; t += step) {
    cp_async_wait<S - 1>();
    __syncwarp();
    const uint64_t b = t * BLOCK + threadIdx.x;
    if (b < nbody) {
      uint4 v[PT];
#pragma unroll
      for (int q = 0; q < PT; ++q) {
        const uint32_t sh = static_cast<uint32_t>(in0(q) & 15u);
        const uint32_t src = sbase + kRank * (slot * PT + q);
        const uint4 lo = ld_shared16(src);
        v[q] = sh ? realign16(lo, ld_shared16(src + 16u), sh) : lo;
      }
      float acc[E];
      fold_vector<DT, ORDER, PT, true>(p, J, 0, v, acc);
      const uint4 y = T::narrow(acc);
      const uint64_t byte_off = (J.head + static_cast<uint64_t>(E) * b) * T::kSize;
      for (uint32_t m = 0; m < J.nout; ++m) {
        uint4* d = reinterpret_cast<uint4*>(out_ptr(p, J, m) + byte_off);
        if (output_ok<DT>(p, J, m, d, 16, kSiteRedStaged)) st16(d, y);
      }
    }
    __syncwarp();
    issue(slot, t_issue);
    t_issue += step;
    slot = (slot + 1 == S) ? 0 : slot + 1;
  }
  cp_async_wait<0>();
}

// The input blocks of body units [b0, b1) of the staged realigning job,
// prefetched into L2 (thread q < P: rank q's span, widened to the 16-byte
// blocks holding its first and last byte).
template <int DT, int MAXJ, int MAXPTR>
__device__ __forceinline__ void realign_prefetch(const ReduceParams<MAXJ, MAXPTR>& p, uint64_t b0,
                                                 uint64_t b1) {
  using T = Elem<DT>;
  const ReduceJob& J = p.job[0];
  if (b0 >= b1 || threadIdx.x >= static_cast<unsigned>(p.P)) return;
  const uint64_t a = reinterpret_cast<uint64_t>(in_ptr(p, J, threadIdx.x)) + (J.in_off + J.head) * T::kSize;
  const uint64_t lo = (a + 16 * b0) & ~static_cast<uint64_t>(15);
  const uint64_t hi = (a + 16 * b1 + 15) & ~static_cast<uint64_t>(15);
  for (uint64_t c = lo; c < hi; c += 32768) {
    const uint64_t n = min(static_cast<uint64_t>(32768), hi - c);
    if (input_ok<DT>(p, J, threadIdx.x, reinterpret_cast<const void*>(c), n, kSiteRedPrefetch))
      prefetch_l2(reinterpret_cast<const void*>(c), static_cast<uint32_t>(n));
  }
}

template <int DT, int MAXJ, int MAXPTR>
__device__ __forceinline__ void reduce_enter(const ReduceParams<MAXJ, MAXPTR>& p, uint64_t tile,
                                             uint64_t first, uint64_t step) {
  pdl_launch_dependents();
  for (int i = 0; i < p.prefetch; ++i)
    reduce_prefetch_tile<DT>(p, tile, first + static_cast<uint64_t>(i) * step);
  pdl_wait();
}

template <int DT, int ORDER, int PT, int MAXJ, int MAXPTR>
__global__ void __launch_bounds__(kReduceBlock)
    dc_reduce_kernel(const __grid_constant__ ReduceParams<MAXJ, MAXPTR> p) {
  constexpr int kUnroll = reduce_unroll(PT);
  const uint64_t tile = static_cast<uint64_t>(p.tile_units);
  reduce_enter<DT>(p, tile, blockIdx.x, gridDim.x);
  reduce_tiles<DT, ORDER, kReduceBlock, kUnroll, PT>(p, tile, blockIdx.x, gridDim.x);
}

// All_reduce of one tensor with realigned inputs (reduce_realign_staged);
// tiles of kReduceBlock body units.
template <int DT, int ORDER, int PT, int MAXJ, int MAXPTR>
__global__ void __launch_bounds__(kReduceBlock, 2)
    dc_reduce_realign_kernel(const __grid_constant__ ReduceParams<MAXJ, MAXPTR> p) {
  pdl_launch_dependents();
  {
    using T = Elem<DT>;
    const ReduceJob& J = p.job[0];
    const uint64_t nbody = (J.count - J.head) / T::kPerVec;
    uint64_t t = blockIdx.x;
    for (int i = 0; i < p.prefetch; ++i, t += gridDim.x)
      realign_prefetch<DT>(p, min(t * kReduceBlock, nbody), min((t + 1) * kReduceBlock, nbody));
  }
  pdl_wait();
  reduce_realign_staged<DT, ORDER, kReduceBlock, PT, kRealignReduceStages>(p, blockIdx.x, gridDim.x);
}

template <int DT, int ORDER, int PT, int MAXJ, int MAXPTR>
__global__ void __launch_bounds__(kReduceSingleBlock)
    dc_reduce_single_kernel(const __grid_constant__ ReduceParams<MAXJ, MAXPTR> p) {
  constexpr int kUnroll = reduce_unroll(PT);
  constexpr uint64_t kTile = static_cast<uint64_t>(kReduceSingleBlock) * kUnroll;
  reduce_enter<DT>(p, kTile, 0, 1);
  reduce_tiles<DT, ORDER, kReduceSingleBlock, kUnroll, PT>(p, kTile, 0, 1);
}

// Kernels that ask for more than 48 KB of dynamic shared memory must say so
// once per device.
template <int DT, int ORDER, int PT, int MAXJ, int MAXPTR>
cudaError_t allow_realign_smem() {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(dc_reduce_realign_kernel<DT, ORDER, PT, MAXJ, MAXPTR>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(realign_reduce_smem(PT)));
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

template <int DT, int ORDER, int PT, int MAXJ, int MAXPTR>
cudaError_t launch_pt(const ReduceParams<MAXJ, MAXPTR>& p, int grid, bool single, bool pdl,
                      cudaStream_t s) {
  if constexpr (PT > 0 && MAXJ == 1) {
    if (!single && p.staged) {  // the planner checked: one job, kJobVec | kJobRealign
      if (p.njobs != 1 || p.job[0].flags != (kJobVec | kJobRealign)) return cudaErrorInvalidValue;
      const cudaError_t e = allow_realign_smem<DT, ORDER, PT, MAXJ, MAXPTR>();
      if (e != cudaSuccess) return e;
      return launch_ex(dc_reduce_realign_kernel<DT, ORDER, PT, MAXJ, MAXPTR>, grid, kReduceBlock, pdl, s,
                       p, realign_reduce_smem(PT));
    }
  }
  if (single)
    return launch_ex(dc_reduce_single_kernel<DT, ORDER, PT, MAXJ, MAXPTR>, 1, kReduceSingleBlock, pdl,
                     s, p);
  if (p.tile_units < 1) return cudaErrorInvalidValue;
  return launch_ex(dc_reduce_kernel<DT, ORDER, PT, MAXJ, MAXPTR>, grid, kReduceBlock, pdl, s, p);
}

template <int DT, int ORDER, int MAXJ, int MAXPTR>
cudaError_t launch_order(const ReduceParams<MAXJ, MAXPTR>& p, int grid, bool single, bool pdl,
                         cudaStream_t s) {
  switch (reduce_pt(p.P)) {
    case 2: return launch_pt<DT, ORDER, 2>(p, grid, single, pdl, s);
    case 4: return launch_pt<DT, ORDER, 4>(p, grid, single, pdl, s);
    case 8: return launch_pt<DT, ORDER, 8>(p, grid, single, pdl, s);
    default: return launch_pt<DT, ORDER, 0>(p, grid, single, pdl, s);
  }
}

template <int DT, int MAXJ, int MAXPTR>
cudaError_t launch_dtype(const ReduceParams<MAXJ, MAXPTR>& p, int order, int grid, bool single,
                         bool pdl, cudaStream_t s) {
  return order == kOrderTree ? launch_order<DT, kOrderTree>(p, grid, single, pdl, s)
                             : launch_order<DT, kOrderLinear>(p, grid, single, pdl, s);
}

template <int DT, int ORDER, int PT, int MAXJ, int MAXPTR>
int occupancy_pt() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, dc_reduce_kernel<DT, ORDER, PT, MAXJ, MAXPTR>, kReduceBlock, 0) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return n > 0 ? n : 1;
}

template <int DT, int ORDER, int PT, int MAXJ, int MAXPTR>
int occupancy_realign_pt() {
  int n = 0;
  cudaError_t e = allow_realign_smem<DT, ORDER, PT, MAXJ, MAXPTR>();
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dc_reduce_realign_kernel<DT, ORDER, PT, MAXJ, MAXPTR>,
                                                      kReduceBlock, realign_reduce_smem(PT));
  if (e != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return n > 0 ? n : 1;
}

template <int DT, int ORDER, int MAXJ, int MAXPTR>
int occupancy_realign_order(int P) {
  switch (reduce_pt(P)) {
    case 2: return occupancy_realign_pt<DT, ORDER, 2, MAXJ, MAXPTR>();
    case 4: return occupancy_realign_pt<DT, ORDER, 4, MAXJ, MAXPTR>();
    default: return occupancy_realign_pt<DT, ORDER, 8, MAXJ, MAXPTR>();
  }
}

template <int DT, int ORDER, int MAXJ, int MAXPTR>
int occupancy_order(int P) {
  switch (reduce_pt(P)) {
    case 2: return occupancy_pt<DT, ORDER, 2, MAXJ, MAXPTR>();
    case 4: return occupancy_pt<DT, ORDER, 4, MAXJ, MAXPTR>();
    case 8: return occupancy_pt<DT, ORDER, 8, MAXJ, MAXPTR>();
    default: return occupancy_pt<DT, ORDER, 0, MAXJ, MAXPTR>();
  }
}

template <int DT, int MAXJ, int MAXPTR>
int occupancy_dtype(int order, int P) {
  return order == kOrderTree ? occupancy_order<DT, kOrderTree, MAXJ, MAXPTR>(P)
                             : occupancy_order<DT, kOrderLinear, MAXJ, MAXPTR>(P);
}

}  // namespace red
}  // namespace dc

// Instantiates the launch and occupancy entry points of one element type.
#define DC_REDUCE_INSTANTIATE(DT, NAME)                                                            \
  namespace dc {                                                                                   \
  cudaError_t launch_reduce_##NAME(const ReduceParams1& p, int order, int grid, bool single,       \
                                   bool pdl, cudaStream_t s) {                                     \
    return red::launch_dtype<DT>(p, order, grid, single, pdl, s);                                  \
  }                                                                                                \
  cudaError_t launch_reduce_##NAME(const ReduceParamsS& p, int order, int grid, bool single,       \
                                   bool pdl, cudaStream_t s) {                                     \
    return red::launch_dtype<DT>(p, order, grid, single, pdl, s);                                  \
  }                                                                                                \
  cudaError_t launch_reduce_##NAME(const ReduceParamsL& p, int order, int grid, bool single,       \
                                   bool pdl, cudaStream_t s) {                                     \
    return red::launch_dtype<DT>(p, order, grid, single, pdl, s);                                  \
  }                                                                                                \
  int reduce_ctas_per_sm_##NAME(int variant, int order, int P) {                                   \
    switch (variant) {                                                                             \
      case 0: return red::occupancy_dtype<DT, 1, 2 * kMaxRanks>(order, P);                        \
      case 1: return red::occupancy_dtype<DT, kMaxRanks, 4 * kMaxRanks>(order, P);                \
      case 3:                                                                                      \
        return order == kOrderTree                                                                 \
                   ? red::occupancy_realign_order<DT, kOrderTree, 1, 2 * kMaxRanks>(P)             \
                   : red::occupancy_realign_order<DT, kOrderLinear, 1, 2 * kMaxRanks>(P);          \
      default: return red::occupancy_dtype<DT, kManyMaxReduceJobs, kManyMaxReducePtrs>(order, P); \
    }                                                                                              \
  }                                                                                                \
  DC_BOUNDS_READER(take_bounds_reduce_##NAME)                                                      \
  }  // namespace dc
