// dc_api.cu -- the C ABI of libdc: argument checks, path planning, launch.
//
// Pages cited by title:
//   [PR491] "perf(cuda): vectorize the deterministic all-gather copy and
//           right-size its single-block path" (RL-Kernel pull request 491).
//
// Planning follows what [PR491] learned on B200 and re-measures it here:
//  * the single-block path only pays below a crossover on OUTPUT bytes for
//    the gather (section "What", kAllGatherSingleBlockMaxBytes) and on INPUT
//    bytes per rank for the reductions (author's reply:
//    input_bytes <= kSingleBlockFastPathMaxBytes); on GB300 the measured
//    crossovers are 0 for one-tensor gathers (but for unaligned jobs under
//    128 B per rank) and reductions, and 16 KiB for all_gather_many; all
//    can be changed at run time;
//  * the multi-block grid is sized from the 16-byte vector (or 8-element
//    group) count, not from bytes (review nitpick on
//    DeterministicCollectiveState::all_gather: a byte-sized grid left 15 of
//    16 blocks idle), capped at the resident CTAs of the whole GPU, and the
//    single-job kernels' tiles are sized so that every SM gets the same
//    share (even_tile).
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "dc.h"
#include "dc_device.cuh"
#include "dc_internal.h"

namespace {

using namespace dc;

thread_local char g_err[512] = "";
std::atomic<unsigned long long> g_launches{0};
thread_local int g_last_grid = 0;  // CTAs of this thread's last launch

// Single-CTA thresholds measured on GB300 (per-call time of back-to-back
// calls in a CUDA graph: 14 calls on distinct buffers after an L2 flush, and
// 200 identical calls with warm caches; a call timed alone after an L2 flush
// reads within one 2 us tick of the event clock for both paths at these
// sizes).  Gather: since the multi-CTA kernel spreads a small output evenly
// over the SMs and loads a single round straight into registers, it is
// faster at every size measured, 2 to 32 KiB of output (2 KiB: 1.42-1.56 vs
// 1.56-1.76 us cold, 0.94-0.99 vs 1.12-1.18 us warm; 16 KiB: 1.56-1.68 vs
// 1.75-1.90 us cold); before those two changes one CTA won up to 16 KiB.
// All_reduce (P = 8): the grid is never slower, from 1 KiB per rank (1.86 vs
// 1.93 us) up.  So the single-CTA kernels run only when forced.
constexpr long long kDefaultGatherSingleMax = 0;
// all_gather_many: one CTA up to 16 KiB of output (4 tensors of 512-2048 B x
// 4 ranks: 2.44 vs 2.93 us cold, 1.73 vs 2.36 us warm; the split launch
// costs more than it spreads).
constexpr long long kDefaultGatherManySingleMax = 16 * 1024;
constexpr long long kDefaultReduceSingleMax = 0;

struct Options {
  std::atomic<long long> force_path{0};
  std::atomic<long long> force_generic{0};
  std::atomic<long long> gather_single_max{kDefaultGatherSingleMax};
  std::atomic<long long> gather_many_single_max{kDefaultGatherManySingleMax};
  std::atomic<long long> reduce_single_max{kDefaultReduceSingleMax};
  std::atomic<long long> grid_ctas{0};
  std::atomic<long long> test_fail_launch{0};
  std::atomic<long long> pdl{1};
  std::atomic<long long> gather_staged{1};
  std::atomic<long long> split_cost_pct{250};       // see plan_split
  std::atomic<long long> split_cost_warp_pct{100};  // see plan_split
  std::atomic<long long> prefetch{1};
  std::atomic<long long> tile_min{512};  // see staged_tile
  std::atomic<long long> reduce_tile_min{64};  // see launch_reduce_plan
  std::atomic<long long> reduce_staged{1};     // see launch_reduce_plan
  std::atomic<long long> gather_bulk{0};       // see plan_bulk
  std::atomic<long long> bulk_min_bytes{0};
  std::atomic<long long> bulk_chunk_bytes{16384};
  std::atomic<long long> bulk_chunk_min{2048};
  std::atomic<long long> bulk_stages{6};
  std::atomic<long long> bulk_ctas_per_sm{2};
  std::atomic<long long> bulk_prefetch{2};
  std::atomic<long long> fused_chunk_min{32768};
  std::atomic<long long> fused_tma{1};
  std::atomic<long long> fused_stages{3};
  std::atomic<long long> fused_sub_bytes{32768};
  std::atomic<long long> realign_warp{1};
  std::atomic<long long> test_fused_absent{0};
  std::atomic<long long> wait_limit_ns{1000000000};
  std::atomic<long long> test_bulk_short_tx{0};
};
Options g_opt;
std::once_flag g_env_once;

struct OptionKey {
  const char* key;
  const char* env;
  std::atomic<long long>* slot;
};
const OptionKey kKeys[] = {
    {"force_path", "DC_FORCE_PATH", &g_opt.force_path},
    {"force_generic", "DC_FORCE_GENERIC", &g_opt.force_generic},
    {"gather_single_max_bytes", "DC_GATHER_SINGLE_MAX_BYTES", &g_opt.gather_single_max},
    {"gather_many_single_max_bytes", "DC_GATHER_MANY_SINGLE_MAX_BYTES", &g_opt.gather_many_single_max},
    {"reduce_single_max_bytes", "DC_REDUCE_SINGLE_MAX_BYTES", &g_opt.reduce_single_max},
    {"grid_ctas", "DC_GRID_CTAS", &g_opt.grid_ctas},
    {"test_fail_launch", nullptr, &g_opt.test_fail_launch},
    {"pdl", "DC_PDL", &g_opt.pdl},
    {"gather_staged", "DC_GATHER_STAGED", &g_opt.gather_staged},
    {"gather_split_cost_pct", "DC_GATHER_SPLIT_COST_PCT", &g_opt.split_cost_pct},
    {"gather_split_cost_warp_pct", "DC_GATHER_SPLIT_COST_WARP_PCT", &g_opt.split_cost_warp_pct},
    {"prefetch", "DC_PREFETCH", &g_opt.prefetch},
    {"gather_tile_min", "DC_GATHER_TILE_MIN", &g_opt.tile_min},
    {"reduce_tile_min", "DC_REDUCE_TILE_MIN", &g_opt.reduce_tile_min},
    {"reduce_staged", "DC_REDUCE_STAGED", &g_opt.reduce_staged},
    {"gather_bulk", "DC_GATHER_BULK", &g_opt.gather_bulk},
    {"gather_bulk_min_bytes", "DC_GATHER_BULK_MIN_BYTES", &g_opt.bulk_min_bytes},
    {"bulk_chunk_bytes", "DC_BULK_CHUNK_BYTES", &g_opt.bulk_chunk_bytes},
    {"bulk_chunk_min", "DC_BULK_CHUNK_MIN", &g_opt.bulk_chunk_min},
    {"bulk_stages", "DC_BULK_STAGES", &g_opt.bulk_stages},
    {"bulk_ctas_per_sm", "DC_BULK_CTAS_PER_SM", &g_opt.bulk_ctas_per_sm},
    {"bulk_prefetch", "DC_BULK_PREFETCH", &g_opt.bulk_prefetch},
    {"fused_chunk_min", "DC_FUSED_CHUNK_MIN", &g_opt.fused_chunk_min},
    {"fused_tma", "DC_FUSED_TMA", &g_opt.fused_tma},
    {"fused_stages", "DC_FUSED_STAGES", &g_opt.fused_stages},
    {"fused_sub_bytes", "DC_FUSED_SUB_BYTES", &g_opt.fused_sub_bytes},
    {"gather_realign_warp", "DC_GATHER_REALIGN_WARP", &g_opt.realign_warp},
    {"test_fused_absent_ranks", nullptr, &g_opt.test_fused_absent},
    {"wait_limit_ns", "DC_WAIT_LIMIT_NS", &g_opt.wait_limit_ns},
    {"test_bulk_short_tx", nullptr, &g_opt.test_bulk_short_tx},
};

void read_env_once() {
  std::call_once(g_env_once, [] {
    for (const OptionKey& k : kKeys) {
      if (!k.env) continue;
      const char* v = std::getenv(k.env);
      if (!v || !*v) continue;
      char* end = nullptr;
      long long x = std::strtoll(v, &end, 0);
      if (end && *end == '\0' && x >= 0) k.slot->store(x);
    }
  });
}

dc_status_t fail(dc_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return s;
}

dc_status_t ok() {
  g_err[0] = '\0';
  return DC_OK;
}

bool overlaps(uint64_t a, uint64_t na, uint64_t b, uint64_t nb) {
  return na > 0 && nb > 0 && a < b + nb && b < a + na;
}

// ---------------------------------------------------- device properties ---
constexpr int kMaxDevices = 64;
constexpr int kFamilies = 128;  // gather: family * kGatherModes + mode (< 18); reductions: 24 + (< 72); staged realigning reduction: 96 + (< 24); fused all-gather: 127
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_occ[kMaxDevices][kFamilies];

dc_status_t current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DC_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  }
  if (*dev < 0 || *dev >= kMaxDevices) return fail(DC_ERR_CUDA, "device index %d out of range", *dev);
  return DC_OK;
}

dc_status_t sm_count(int dev, int* sms) {
  int v = g_sms[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    cudaError_t e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || v <= 0) {
      cudaGetLastError();
      return fail(DC_ERR_CUDA, "cannot read the SM count: %s", cudaGetErrorString(e));
    }
    g_sms[dev].store(v, std::memory_order_relaxed);
  }
  *sms = v;
  return DC_OK;
}

template <class F>
int occupancy(int dev, int family, F query) {
  int v = g_occ[dev][family].load(std::memory_order_relaxed);
  if (v <= 0) {
    v = std::max(1, query());
    g_occ[dev][family].store(v, std::memory_order_relaxed);
  }
  return v;
}

// Multi-CTA grid for `tiles` tiles of work taken round robin: at most the
// CTAs that fit on the GPU at once (less `reserve` kept for other CTAs of the
// launch), and the fewest CTAs that still finish in the same number of rounds
// (so every CTA does the same number of tiles, give or take one).
int plan_grid(uint64_t tiles, int sms, int ctas_per_sm, int reserve = 0) {
  const uint64_t all = static_cast<uint64_t>(sms) * static_cast<uint64_t>(ctas_per_sm);
  const uint64_t cap = std::max<uint64_t>(1, all > static_cast<uint64_t>(reserve) ? all - reserve : 1);
  if (tiles == 0) return 1;  // (a launch with only scalar head and tail work)
  uint64_t g;
  const long long forced = g_opt.grid_ctas.load();
  if (forced > 0) {
    g = std::min<uint64_t>(static_cast<uint64_t>(forced), std::max<uint64_t>(tiles, 1));
  } else {
    const uint64_t rounds = (tiles + cap - 1) / cap;
    g = std::max<uint64_t>(1, (tiles + rounds - 1) / std::max<uint64_t>(rounds, 1));
  }
  return static_cast<int>(std::min<uint64_t>(g, 0x7FFFFFFFull));
}

bool use_single(uint64_t size_bytes, long long threshold) {
  const long long f = g_opt.force_path.load();
  if (f == 1) return true;
  if (f == 2) return false;
  return size_bytes <= static_cast<uint64_t>(threshold);
}

dc_status_t check_launch(cudaError_t e, const char* what, int grid) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DC_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
  }
  g_launches.fetch_add(1, std::memory_order_relaxed);
  g_last_grid = grid;
  return ok();
}

// --------------------------------------------------------------- gather ---
struct GatherTensor {
  uint64_t out;
  uint64_t bytes;
  const void* const* peers;  // P pointers
};

bool tensor_aligned(const GatherTensor& g, int P, bool allow_flat) {
  bool aligned = allow_flat && (g.out & 15u) == 0 && (g.bytes & 15u) == 0;
  for (int r = 0; r < P && aligned; ++r)
    aligned = (reinterpret_cast<uint64_t>(g.peers[r]) & 15u) == 0;
  return aligned;
}

// Rejects an output of a batch of gathers that overlaps another output or any
// payload (payloads may overlap each other).  The T outputs and T*P payloads
// are sorted by start and swept once, keeping per kind (output, payload) the
// range that reaches furthest so far: since every earlier range starts at or
// before the current one, the current range overlaps an earlier range of a
// kind exactly when that kind's furthest end lies past its start.
// O(n log n) for the n = T*(P+1) ranges of a call.
dc_status_t check_gather_overlaps(const GatherTensor* ts, int T, int P) {
  struct R {
    uint64_t lo, hi;
    int t, r;  // r < 0: the output of tensor t
  };
  std::vector<R> v;
  v.reserve(static_cast<size_t>(T) * (P + 1));
  for (int t = 0; t < T; ++t) {
    const uint64_t B = ts[t].bytes;
    if (B == 0) continue;
    v.push_back(R{ts[t].out, ts[t].out + B * static_cast<uint64_t>(P), t, -1});
    for (int r = 0; r < P; ++r) {
      const uint64_t s = reinterpret_cast<uint64_t>(ts[t].peers[r]);
      v.push_back(R{s, s + B, t, r});
    }
  }
  std::sort(v.begin(), v.end(), [](const R& a, const R& b) { return a.lo < b.lo; });
  const R* far_out = nullptr;  // the output reaching furthest so far
  const R* far_in = nullptr;   // the payload reaching furthest so far
  for (const R& x : v) {
    if (x.r < 0) {
      if (far_out && far_out->hi > x.lo)
        return fail(DC_ERR_OVERLAP, "outputs of tensors %d and %d overlap", std::min(far_out->t, x.t),
                    std::max(far_out->t, x.t));
      if (far_in && far_in->hi > x.lo)
        return fail(DC_ERR_OVERLAP, "output of tensor %d overlaps the payload of tensor %d rank %d", x.t,
                    far_in->t, far_in->r);
      if (!far_out || x.hi > far_out->hi) far_out = &x;
    } else {
      if (far_out && far_out->hi > x.lo)
        return fail(DC_ERR_OVERLAP, "output of tensor %d overlaps the payload of tensor %d rank %d",
                    far_out->t, x.t, x.r);
      if (!far_in || x.hi > far_in->hi) far_in = &x;
    }
  }
  return DC_OK;
}

// Fill jobs and sources of a gather parameter block from T tensors.  The
// aligned jobs come first (their vectors are [0, flat_vec)), then the other
// jobs of at least kGatherSmallBytes per rank, then the smaller ones (vectors
// [small_vec, total_vec)); each keeps its own output, so the order changes no
// result.
template <class Params>
void fill_gather(Params& prm, const GatherTensor* ts, int T, int P, bool allow_flat) {
  uint64_t v = 0;
  int nj = 0;
  prm.small_vec = 0;
  prm.small_job0 = 0;
  for (int pass = 0; pass < 3; ++pass) {
    if (pass == 2) {
      prm.small_vec = v;
      prm.small_job0 = nj;
    }
    for (int t = 0; t < T; ++t) {
      const GatherTensor& g = ts[t];
      if (g.bytes == 0) continue;
      const bool aligned = tensor_aligned(g, P, allow_flat);
      const int kind = aligned ? 0 : g.bytes < kGatherSmallBytes ? 2 : 1;
      if (kind != pass) continue;
      GatherJob& J = prm.job[nj];
      J.out = g.out;
      J.bytes = g.bytes;
      J.src0 = static_cast<uint32_t>(nj * P);
      for (int r = 0; r < P; ++r) prm.src[nj * P + r] = reinterpret_cast<uint64_t>(g.peers[r]);
      J.flags = aligned ? kJobFlat : (g.bytes < kGatherSmallBytes ? kJobSmall : 0u);
      const uint64_t end = g.out + static_cast<uint64_t>(P) * g.bytes;
      J.nvec = ((end - 1) >> 4) - (g.out >> 4) + 1;
      J.vfirst = v;
      v += J.nvec;
      ++nj;
    }
    if (pass == 0) prm.flat_vec = v;
  }
  prm.njobs = nj;
  prm.P = P;
  prm.total_vec = v;
}

// Split of a launch's CTAs (at most `cap`) between its three parts: the
// jobs of fewer than kGatherSmallBytes per rank get one CTA per kGatherBlock
// threads, kSmallSplit threads per output vector (so all their byte loads
// are in flight at once), at most kMaxSmallCtas, at the end of the grid, each
// CTA a contiguous run of small_per vectors whose first and last jobs
// small_tab records; the rest goes to the
// aligned jobs (tiles of kSplitVectors vectors per thread) and the other
// unaligned jobs (tiles of kSplitRealignVectors), in proportion to their
// work: a realigned 16-byte vector counts gather_split_cost_pct / 100 staged
// ones, so both parts finish together.  Measured on GB300 with the six mixed
// tensors of the all_gather_many workload (P = 8), both parts staged: 100 %
// -> 115 us, 150 % -> 108.5 us, 200 % -> 108 us, 250 % -> 100.6 us, 300 %
// -> 104 us; every CTA on the register realigning path instead: 141 us.
// A realigning part of more than kRoundRobinJobs jobs realigns across the
// lanes of a warp instead (gather_realign_warp on), with boundary CTAs for
// its rank-boundary vectors, and its vectors count
// gather_split_cost_warp_pct / 100 staged ones.  Measured (20 calls back to
// back, payloads of every other tensor at +1 B; ring at 250 % -> warp at 250
// % / 100 %): 60 tensors x 8 ranks of 1-128 KiB 13.3 -> 13.3 / 10.8 us, 100
// x 8 of 16 B-64 KiB 11.6 -> 11.3 / 9.7 us; all unaligned, 250 x 4 of 4-64
// KiB 17.3 -> 11.6 us, 60 x 8 of 1-128 KiB 13.3 -> 9.8 us.  The six mixed
// tensors (one unaligned job of 7 MiB+5 B) stay on the ring: on the warp path
// they took 113-114 us against 109 us.
// Each part gets the fewest CTAs that finish its tiles in the same number of
// rounds.  Returns the total grid, 0 if no split is possible (fewer CTAs than
// parts with work).
// Parts of all_gather_many with more jobs than this take contiguous runs
// of tiles per CTA (and the realigning part realigns across warps).
constexpr int kRoundRobinJobs = 16;

template <class Params>
int plan_split(Params& prm, uint64_t cap) {
  const uint64_t fv = prm.flat_vec, gv = prm.small_vec - prm.flat_vec, sv = prm.total_vec - prm.small_vec;
  const uint64_t others = (fv > 0 ? 1 : 0) + (gv > 0 ? 1 : 0);
  if (cap < others + (sv > 0 ? 1 : 0)) return 0;
  constexpr size_t kTab = sizeof(prm.small_tab) / sizeof(prm.small_tab[0]);
  uint64_t sc = 0;
  if (sv > 0) {
    if (kTab < 2) return 0;  // (parameter blocks of one job have no small-job part)
    // one CTA per kGatherBlock / kSmallSplit vectors, each CTA a contiguous run
    sc = std::min<uint64_t>({(sv * kSmallSplit + kGatherBlock - 1) / kGatherBlock, cap - others,
                             static_cast<uint64_t>(kTab - 1)});
    const uint64_t per = (sv + sc - 1) / sc;
    sc = (sv + per - 1) / per;
    prm.small_per = static_cast<uint32_t>(per);
    // small_tab[c]: the job of CTA c's first vector; small_tab[sc]: the last job
    int j = prm.small_job0;
    for (uint64_t c = 0; c < sc; ++c) {
      const uint64_t v = prm.small_vec + c * per;
      while (j + 1 < prm.njobs && prm.job[j + 1].vfirst <= v) ++j;
      prm.small_tab[c] = static_cast<uint16_t>(j - prm.small_job0);
    }
    prm.small_tab[sc] = static_cast<uint16_t>(prm.njobs - 1 - prm.small_job0);
  }
  cap -= sc;
  // the realigning part: across warps (with CTAs for its jobs' rank-boundary
  // vectors, one per kGatherBlock (job, boundary) pairs, at most
  // kMaxBoundaryCtas) when it has more than kRoundRobinJobs jobs, else the ring
  int nflat = 0;
  while (nflat < prm.njobs && (prm.job[nflat].flags & kJobFlat)) ++nflat;
  const int nreal = prm.small_job0 - nflat;
  uint64_t bc = 0;
  prm.realign_warp = prm.realign_warp && gv > 0 && nreal > kRoundRobinJobs ? 1 : 0;
  if (prm.realign_warp) {
    const uint64_t pairs = static_cast<uint64_t>(nreal) * static_cast<uint64_t>(prm.P + 1);
    bc = std::min<uint64_t>((pairs + kGatherBlock - 1) / kGatherBlock, kMaxBoundaryCtas);
    if (cap < others + bc) return 0;
    cap -= bc;
  }
  const uint64_t ftile = static_cast<uint64_t>(kGatherBlock) * kSplitVectors;
  const uint64_t gtile = static_cast<uint64_t>(kGatherBlock) * kSplitRealignVectors;
  const uint64_t ft = (fv + ftile - 1) / ftile, gt = (gv + gtile - 1) / gtile;
  uint64_t gf, gg;
  if (gt == 0) {
    gf = std::min(cap, ft);
    gg = 0;
  } else if (ft == 0) {
    gf = 0;
    gg = std::min(cap, gt);
  } else {
    const long long pct = prm.realign_warp ? g_opt.split_cost_warp_pct.load() : g_opt.split_cost_pct.load();
    const double cost = static_cast<double>(std::max(1LL, pct)) / 100.0;
    const double wf = static_cast<double>(fv), wg = cost * static_cast<double>(gv);
    gf = static_cast<uint64_t>(static_cast<double>(cap) * wf / (wf + wg) + 0.5);
    gf = std::min(std::max<uint64_t>(gf, 1), cap - 1);
    gg = cap - gf;
  }
  auto trim = [](uint64_t tiles, uint64_t g) {
    if (g == 0) return g;
    const uint64_t rounds = (tiles + g - 1) / g;
    return (tiles + rounds - 1) / rounds;
  };
  gf = trim(ft, std::min(gf, ft));
  gg = trim(gt, std::min(gg, gt));
  // The aligned and the realigning part each deal their tiles over their
  // CTAs (at most kMaxPartCtas): with more than kRoundRobinJobs jobs every
  // CTA takes a contiguous run of `per` tiles (per_out = per), so that its
  // threads enter only the jobs of that run; with fewer, tiles go round
  // robin (per_out = 0).  Measured on GB300: 250 tensors x 4 ranks of 128
  // B-4 KiB at +1 B 36.0 -> 5.3 us with runs, 4-64 KiB aligned 38.1 -> 9.9
  // us; the six-tensor batch (8 x 32 MiB in it) 2-3 % slower with runs than
  // round robin.  tab[c] is the job of CTA c's first vector, found by one
  // forward walk over the jobs.
  constexpr uint64_t kPartTab = sizeof(prm.flat_tab) / sizeof(prm.flat_tab[0]);
  auto deal = [&](uint64_t tiles, uint64_t g, uint64_t tile, uint64_t v0, int njobs_part, uint16_t* tab,
                     uint32_t* per_out) {
    if (g == 0 || tiles == 0) {
      *per_out = 0;
      return static_cast<uint64_t>(0);
    }
    uint64_t per = 0;
    if (njobs_part > kRoundRobinJobs) {
      per = (tiles + g - 1) / g;
      if ((tiles + per - 1) / per > kPartTab) per = (tiles + kPartTab - 1) / kPartTab;
      g = (tiles + per - 1) / per;
    } else {
      g = std::min<uint64_t>(g, kPartTab);
    }
    *per_out = static_cast<uint32_t>(per);
    int j = 0;
    for (uint64_t c = 0; c < g; ++c) {
      const uint64_t v = v0 + c * (per ? per : 1) * tile;
      while (j + 1 < prm.njobs && prm.job[j + 1].vfirst <= v) ++j;
      tab[c] = static_cast<uint16_t>(j);
    }
    return g;
  };
  gf = deal(ft, gf, ftile, 0, nflat, prm.flat_tab, &prm.flat_per);
  gg = deal(gt, gg, gtile, fv, nreal, prm.real_tab, &prm.real_per);
  prm.flat_ctas = static_cast<int32_t>(gf);
  prm.small_ctas = static_cast<int32_t>(sc);
  prm.bnd_ctas = static_cast<int32_t>(gg ? bc : 0);
  return static_cast<int>(gf + gg + prm.bnd_ctas + sc);
}

// Work units per tile, chosen so that every SM gets the same share of a
// launch's units: a CTA moves its tiles through one SM's load and store ports,
// and a call is over when its busiest SM is.  A launch of more than one full
// tile per resident CTA (sms * occ of them) takes R = ceil(total / (sms * occ
// * full)) rounds of tiles of total / (sms * occ * R) units.  A smaller one
// is cut into tiles of about total / (sms * k) units, with k the most CTAs
// per SM (up to occ) that keep a tile at `min_tile` units or more.  Tiles are
// rounded up to a multiple of `gran` units: 32 where every unit is a 16-byte
// aligned load or store, so that each warp access covers whole 128-byte
// lines (the 8627x8192 all_reduce took 7 % longer with tiles of 510 units
// than of 512); 2 for the realigning gather, whose loads are not aligned
// anyway and where rounding to 32 left CTA slots empty (8 x (32 MiB+1): 37
// rounds of 1024-vector tiles on 443 CTAs instead of 998-vector tiles on
// 455).  `reserve` CTA slots are kept for other CTAs of the launch.
uint64_t even_tile(uint64_t total, int sms, int occ, uint64_t full, long long min_tile, uint64_t gran,
                   int reserve = 0) {
  const uint64_t lo = std::min<uint64_t>(full, static_cast<uint64_t>(std::max(32LL, min_tile)));
  const uint64_t nsm = static_cast<uint64_t>(std::max(sms, 1));
  const uint64_t all = nsm * static_cast<uint64_t>(std::max(occ, 1));
  const uint64_t slots = all > static_cast<uint64_t>(reserve) ? all - reserve : 1;
  if (total > slots * full) {  // several rounds: every CTA the same number of equal tiles
    const uint64_t rounds = (total + slots * full - 1) / (slots * full);
    const uint64_t per = slots * rounds;
    return std::min(full, ((total + per - 1) / per + gran - 1) / gran * gran);
  }
  for (int k = std::max(occ, 1); k >= 1; --k) {
    const uint64_t per = std::min(slots, nsm * static_cast<uint64_t>(k));
    const uint64_t t = ((total + per - 1) / per + gran - 1) / gran * gran;
    if (t >= lo) return std::min(full, t);
  }
  return lo;
}

template <class Params>
dc_status_t launch_gather_plan(Params& prm, int family, uint64_t out_bytes, cudaStream_t stream) {
  if (g_opt.test_fail_launch.load())
    return fail(DC_ERR_CUDA, "launch failure injected by the test_fail_launch option");
  int dev = 0, sms = 0;
  dc_status_t st = current_device(&dev);
  if (st != DC_OK) return st;
  st = sm_count(dev, &sms);
  if (st != DC_OK) return st;
  // One tensor: the grid, except a job under kGatherSmallBytes per rank (at
  // most 8 KiB of output), whose vectors are all byte-assembled and which
  // one CTA copies with each vector's loads issued first (P = 8 x 100 B at
  // +1 B: 5.9 us on the multi-CTA kernel, whose byte path has no registers to
  // spare).  Batches: one CTA up to gather_many_single_max_bytes of output.
  const bool small_job = family == 0 && (prm.job[0].flags & kJobSmall) != 0;
  const bool single =
      use_single(out_bytes, small_job ? (1LL << 62)
                                      : family == 0 ? g_opt.gather_single_max.load()
                                                    : g_opt.gather_many_single_max.load());
  prm.staged = g_opt.gather_staged.load() ? 1 : 0;
  prm.realign_warp = g_opt.realign_warp.load() ? 1 : 0;
  prm.prefetch = static_cast<int32_t>(std::min<long long>(g_opt.prefetch.load(), 64));
  prm.flat_ctas = 0;
  prm.small_ctas = 0;
  prm.bnd_ctas = 0;
  prm.tile_vec = 0;  // single-CTA launches: the kernel's own tile
  int grid = 1;
  if (!single) {
    int mode = gather_mode_of(prm);
    if (mode == kGatherModeSplit) {
      const int occ = occupancy(dev, family * kGatherModes + mode,
                                [family, mode] { return gather_ctas_per_sm(family, mode); });
      const long long forced = g_opt.grid_ctas.load();
      const uint64_t cap = forced > 0 ? static_cast<uint64_t>(forced)
                                      : static_cast<uint64_t>(sms) * static_cast<uint64_t>(occ);
      grid = plan_split(prm, std::min<uint64_t>(cap, 0x7FFFFFFFull));
      if (grid == 0) {  // fewer CTAs than parts: every CTA takes the realigning path
        prm.staged = 0;
        prm.flat_ctas = 0;
        prm.small_ctas = 0;
        prm.bnd_ctas = 0;
        mode = gather_mode_of(prm);
      }
    }
    if (mode != kGatherModeSplit) {
      const int fam = family * kGatherModes + mode;
      const int occ = occupancy(dev, fam, [family, mode] { return gather_ctas_per_sm(family, mode); });
      const int unroll = mode == 0   ? kGatherUnrollGeneral
                         : mode == 3 ? kStagedVectors
                         : mode == 5 ? kRealignVectors
                         : mode == 6 ? kWarpRealignVectors
                                     : kGatherUnroll;
      uint64_t tile = static_cast<uint64_t>(kGatherBlock) * unroll;
      // The staged single-job kernels take even tiles: the aligned one (mode
      // 3) of at least gather_tile_min vectors, the realigning one (mode 5)
      // only when it has several rounds of full tiles.  Measured on GB300 (14
      // calls back to back after an L2 flush, per call; fixed full tiles ->
      // even tiles), aligned: 8 x 8 KiB 2.01 -> 1.74 us, 2 x 1 MiB 2.32 ->
      // 2.16 us, 8 x 1 MiB 3.78 -> 3.48 us, 8 x 2 MiB 6.56 -> 5.83 us, 8 x 4
      // MiB 11.2 -> 10.8 us; 256 tiles of 512 vectors for 2 MiB of output
      // (uneven over 152 SMs) took 2.46 us, and tiles under 512 vectors were
      // slower for outputs of 512 KiB to 2 MiB.  Realigning (payloads at +1 B,
      // output at +3 B, 12 calls): 8 x (1 MiB+1) 7.17 -> 6.63 us, 8 x (2
      // MiB+1) 9.44 -> 8.67 us, 8 x (4 MiB+1) 13.7 -> 13.05 us, whereas
      // smaller tiles in a single round made 8 x (256 KiB+1) and 3 x (1
      // MiB+1) 3-6 % slower.  Mode 5 with 64-bit indices keeps full tiles.
      // Mode 5 adds one CTA for the rank-boundary vectors (copy_boundaries),
      // and keeps a slot free for it.
      // Mode 6 (one unaligned job realigned across warps, registers) takes
      // even tiles of at least gather_tile_min vectors, whole warps each.
      const int reserve = (mode == 5 || mode == 6) ? 1 : 0;
      const bool wide = mode == 5 && (prm.total_vec * 16 >= (1ull << 32) || prm.job[0].bytes >= (1ull << 32));
      if ((mode == 2 || mode == 3 || mode == 5 || mode == 6) && !wide)
        tile = even_tile(prm.total_vec, sms, occ, tile,
                         mode == 5 ? static_cast<long long>(tile) : g_opt.tile_min.load(), mode == 5 ? 2 : 32,
                         reserve);
      if (mode == 2 || mode == 3 || mode == 5 || mode == 6) prm.tile_vec = static_cast<int32_t>(tile);
      grid = plan_grid((prm.total_vec + tile - 1) / tile, sms, occ, reserve) + reserve;
    }
  }
  return check_launch(launch_gather(prm, grid, single, g_opt.pdl.load() != 0, stream), "all-gather",
                      single ? 1 : grid);
}

// One 16-byte aligned gather on the TMA engine (dc_bulk.cu).  Chunks: with
// more than one full chunk (bulk_chunk_bytes) per CTA slot (SMs x
// bulk_ctas_per_sm), R = ceil(total / (slots x full)) rounds of equal chunks
// of total / (slots x R) bytes; a smaller output is cut into chunks of at
// least bulk_chunk_min bytes, one per CTA.  Chunks are rounded up to 128
// bytes (whole L2 lines; rounding up only lowers the chunk count, so no CTA
// gets an extra round).  The ring has bulk_stages stages, fewer when a CTA
// has fewer chunks, and never more than fit kBulkMaxSmem.
struct BulkPlan {
  uint64_t chunk;
  int stages;
  int grid;
};

BulkPlan plan_bulk(uint64_t total, int sms) {
  const uint64_t cps = static_cast<uint64_t>(std::min(std::max(g_opt.bulk_ctas_per_sm.load(), 1LL), 32LL));
  const uint64_t full = std::max<uint64_t>(16, static_cast<uint64_t>(g_opt.bulk_chunk_bytes.load()) & ~15ull);
  const uint64_t cmin = std::min(full, std::max<uint64_t>(16, static_cast<uint64_t>(g_opt.bulk_chunk_min.load())));
  const uint64_t slots = static_cast<uint64_t>(std::max(sms, 1)) * cps;
  auto round_up = [](uint64_t x, uint64_t g) { return (x + g - 1) / g * g; };
  uint64_t chunk;
  if (total > slots * full) {
    const uint64_t rounds = (total + slots * full - 1) / (slots * full);
    chunk = (total + slots * rounds - 1) / (slots * rounds);
  } else {
    const uint64_t g = std::max<uint64_t>(1, std::min(slots, total / cmin));
    chunk = (total + g - 1) / g;
  }
  chunk = chunk >= 128 ? round_up(chunk, 128) : round_up(chunk, 16);
  const uint64_t nchunks = (total + chunk - 1) / chunk;
  const uint64_t grid = std::min<uint64_t>(nchunks, slots);
  const uint64_t per_cta = (nchunks + grid - 1) / grid;
  uint64_t S = std::min<uint64_t>(std::max(g_opt.bulk_stages.load(), 1LL), 32);
  S = std::min(S, per_cta);
  const uint64_t fit = kBulkMaxSmem / (chunk + 8);
  S = std::max<uint64_t>(1, std::min(S, fit));
  const long long forced = g_opt.grid_ctas.load();
  const uint64_t g = forced > 0 ? std::min<uint64_t>(static_cast<uint64_t>(forced), nchunks) : grid;
  return BulkPlan{chunk, static_cast<int>(S), static_cast<int>(std::min<uint64_t>(g, 0x7FFFFFFFull))};
}

dc_status_t launch_bulk_plan(const GatherTensor& t, int P, uint64_t total, cudaStream_t stream) {
  if (g_opt.test_fail_launch.load())
    return fail(DC_ERR_CUDA, "launch failure injected by the test_fail_launch option");
  int dev = 0, sms = 0;
  dc_status_t st = current_device(&dev);
  if (st != DC_OK) return st;
  st = sm_count(dev, &sms);
  if (st != DC_OK) return st;
  BulkParams bp{};
  bp.out = t.out;
  bp.bytes = t.bytes;
  bp.total = total;
  bp.P = P;
  for (int r = 0; r < P; ++r) bp.src[r] = reinterpret_cast<uint64_t>(t.peers[r]);
  const BulkPlan plan = plan_bulk(total, sms);
  bp.chunk = plan.chunk;
  bp.stages = plan.stages;
  // L2 prefetch distance in chunks per CTA, at most 64 MB ahead over the grid
  const uint64_t pf_cap = (64ull << 20) / (plan.chunk * static_cast<uint64_t>(plan.grid));
  bp.prefetch = g_opt.prefetch.load()
                    ? static_cast<int32_t>(std::min<uint64_t>(
                          std::min<uint64_t>(static_cast<uint64_t>(g_opt.bulk_prefetch.load()), 1024),
                          std::max<uint64_t>(pf_cap, 1)))
                    : 0;
  bp.wait_ns = static_cast<uint64_t>(std::max(g_opt.wait_limit_ns.load(), 1000LL));
  bp.test_flags = g_opt.test_bulk_short_tx.load() ? kBulkTestShortTx : 0u;
  return check_launch(launch_gather_bulk(bp, plan.grid, g_opt.pdl.load() != 0, stream), "all-gather (bulk)",
                      plan.grid);
}

// --------------------------------------------------------------- reduce ---
int esize_of(int dtype) { return dtype == kF32 ? 4 : 2; }
int epv_of(int dtype) { return dtype == kF32 ? 4 : 8; }  // elements per 16-byte vector

const char* dtype_name(int dtype) {
  return dtype == kF16 ? "FP16" : dtype == kF32 ? "FP32" : "BF16";
}

// A byte range of one tensor's input or output of rank `rank`.
struct Range {
  uint64_t lo, hi;
  int tensor, rank;
  bool out;
};

// Reject any overlap between an output and another output, and between an
// output and an input unless it is the exact in-place alias of that output:
// all_reduce out_r == in_q (same tensor); reduce_scatter out_r == in_q +
// r * shard bytes (same tensor).  Inputs may overlap inputs.
dc_status_t check_reduce_overlaps(std::vector<Range>& v, bool scatter, const uint64_t* shard_bytes) {
  std::sort(v.begin(), v.end(), [](const Range& x, const Range& y) { return x.lo < y.lo; });
  for (size_t i = 0; i < v.size(); ++i) {
    for (size_t k = i + 1; k < v.size() && v[k].lo < v[i].hi; ++k) {
      const Range& a = v[i];
      const Range& b = v[k];
      if (!a.out && !b.out) continue;
      if (a.out && b.out)
        return fail(DC_ERR_OVERLAP, "outputs of tensor %d rank %d and tensor %d rank %d overlap",
                    a.tensor, a.rank, b.tensor, b.rank);
      const Range& o = a.out ? a : b;
      const Range& in = a.out ? b : a;
      const uint64_t alias = in.lo + (scatter ? static_cast<uint64_t>(o.rank) * shard_bytes[o.tensor] : 0);
      if (o.tensor == in.tensor && o.lo == alias) continue;  // exact in-place alias
      return fail(DC_ERR_OVERLAP,
                  "output of tensor %d rank %d overlaps input %d of tensor %d without being %s",
                  o.tensor, o.rank, in.rank, in.tensor,
                  scatter ? "its own shard of it" : "the same buffer");
    }
  }
  return DC_OK;
}

// A job's units: 16-byte units anchored at its outputs need every output at
// the same address mod 16; inputs at that offset too load whole vectors,
// inputs at other offsets are realigned.  Outputs that disagree: one element
// per unit.  Sets head, flags and nunits of J (in0, out0, nout, in_off and
// count already set); returns nunits.
template <class Params>
uint64_t classify_reduce_job(const Params& prm, ReduceJob& J, int P, int dtype) {
  const int es = esize_of(dtype), epv = epv_of(dtype);
  const uint64_t n = J.count;
  const uint64_t off = J.in_off * es;
  const uint32_t o = static_cast<uint32_t>(prm.ptr[J.out0] & 15u);
  bool outs_agree = true, ins_agree = true;
  for (int m = 0; m < J.nout; ++m) outs_agree = outs_agree && (prm.ptr[J.out0 + m] & 15u) == o;
  for (int q = 0; q < P; ++q) ins_agree = ins_agree && ((prm.ptr[J.in0 + q] + off) & 15u) == o;
  if (outs_agree) {
    uint64_t head = ((16u - o) & 15u) / es;
    if (head > n) head = n;
    const uint64_t rest = n - head;
    J.head = static_cast<uint8_t>(head);
    J.flags = ins_agree ? kJobVec : (kJobVec | kJobRealign);
    J.nunits = (head ? 1 : 0) + rest / epv + ((rest % epv) ? 1 : 0);
  } else {
    J.head = 0;
    J.flags = 0;
    J.nunits = n;
  }
  return J.nunits;
}

template <class Params>
void fill_reduce(Params& prm, int P, int dtype, bool scatter, const std::vector<int>& live,
                 const void* const* in_ptrs, void* const* out_ptrs, const size_t* counts) {
  const int nz = static_cast<int>(live.size());
  prm.P = P;
  for (int k = 0; k < nz; ++k) {
    const int t = live[k];
    for (int q = 0; q < P; ++q) {
      prm.ptr[k * P + q] = reinterpret_cast<uint64_t>(in_ptrs[static_cast<size_t>(t) * P + q]);
      prm.ptr[nz * P + k * P + q] = reinterpret_cast<uint64_t>(out_ptrs[static_cast<size_t>(t) * P + q]);
    }
  }
  uint64_t units = 0;
  int nj = 0;
  for (int k = 0; k < nz; ++k) {
    const uint64_t n = counts[live[k]];
    const int nparts = scatter ? P : 1;
    for (int r = 0; r < nparts; ++r) {
      ReduceJob& J = prm.job[nj++];
      J.in0 = static_cast<uint16_t>(k * P);
      J.out0 = static_cast<uint16_t>(nz * P + k * P + (scatter ? r : 0));
      J.nout = static_cast<uint16_t>(scatter ? 1 : P);
      J.in_off = scatter ? static_cast<uint64_t>(r) * n : 0;
      J.count = n;
      J.ufirst = units;
      units += classify_reduce_job(prm, J, P, dtype);
    }
  }
  prm.njobs = nj;
  prm.total_units = units;
}

template <class Params>
dc_status_t launch_reduce_plan(Params& prm, int variant, int dtype, int order,
                               uint64_t in_bytes_per_rank, cudaStream_t stream, const char* what) {
  if (g_opt.test_fail_launch.load())
    return fail(DC_ERR_CUDA, "launch failure injected by the test_fail_launch option");
  int dev = 0, sms = 0;
  dc_status_t st = current_device(&dev);
  if (st != DC_OK) return st;
  st = sm_count(dev, &sms);
  if (st != DC_OK) return st;
  const bool single = use_single(in_bytes_per_rank, g_opt.reduce_single_max.load());
  prm.prefetch = static_cast<int32_t>(std::min<long long>(g_opt.prefetch.load(), 64));
  prm.tile_units = kReduceBlock * reduce_unroll(reduce_pt(prm.P));
  prm.staged = 0;
  int grid = 1;
  const int pt = reduce_pt(prm.P);
  const int pti = pt == 2 ? 1 : pt == 4 ? 2 : pt == 8 ? 3 : 0;
  // An all_reduce of one tensor whose inputs do not all share the outputs'
  // offset mod 16, P = 2, 4 or 8: the staged realigning kernel, one unit per
  // thread per tile (tiles of kReduceBlock body units).
  if (!single && variant == 0 && pt > 0 && prm.njobs == 1 &&
      prm.job[0].flags == (kJobVec | kJobRealign) && g_opt.reduce_staged.load()) {
    const int P = prm.P;
    const int occ = occupancy(dev, 96 + (dtype * 2 + order) * 4 + pti,
                              [dtype, order, P] { return reduce_ctas_per_sm(dtype, 3, order, P); });
    const int epv = 16 / esize_of(dtype);
    const uint64_t nbody = (prm.job[0].count - prm.job[0].head) / static_cast<uint64_t>(epv);
    prm.staged = 1;
    grid = plan_grid((nbody + kReduceBlock - 1) / kReduceBlock, sms, occ);
  } else if (!single) {
    const int P = prm.P;
    const int fam = 24 + (((dtype * 3 + variant) * 2 + order) * 4 + pti);
    const int occ = occupancy(dev, fam, [dtype, variant, order, P] {
      return reduce_ctas_per_sm(dtype, variant, order, P);
    });
    // One job (an all_reduce of one tensor): tiles spread evenly over the
    // SMs.  Several jobs (reduce_scatter, batches): full tiles, which do not
    // cut a job of a multiple of 512 units; a tile that straddles two jobs
    // runs their parts one after the other, and for 8 shards of 64 Ki BF16
    // elements even tiles were slower (3.70 -> 4.04 us back to back) -- except
    // launches of at most kEvenJobsMaxUnits units, which take even tiles of
    // >= 64 units too, so that a small reduce_scatter reaches more than a few
    // SMs.  Measured (P = 8 BF16 reduce_scatter, 14 calls back to back, per
    // call; full -> even): 128 KiB per rank 3.35 -> 2.90 us, 256 KiB 3.36 ->
    // 3.03 us, 512 KiB 3.48 -> 3.04 us; but 1 MiB 3.77 -> 3.92 us and 8 MiB
    // 13.8 -> 14.9 us, hence the bound.
    // Measured on GB300 for one all_reduce (BF16, 12 calls back to back after
    // an L2 flush, per call; full tiles -> even tiles of >= 64 units): P = 8
    // x 8 KiB 3.36 -> 2.53 us, 8 x 256 KiB 3.56 -> 2.70 us, 8 x 512 KiB 4.21
    // -> 3.01 us, 8 x 2 MiB 6.64 -> 6.11 us, 8 x 8 MiB unchanged; P = 2 x 512
    // KiB 3.97 -> 2.51 us; P = 4 x 2 MiB 5.09 -> 3.88 us.  A 32-unit minimum
    // was no better, 128 and 256 were slower for 128-512 KiB per rank.
    const uint64_t full = static_cast<uint64_t>(kReduceBlock) * reduce_unroll(pt);
    constexpr uint64_t kEvenJobsMaxUnits = 32768;
    const uint64_t tile = prm.njobs == 1 || prm.total_units <= kEvenJobsMaxUnits
                              ? even_tile(prm.total_units, sms, occ, full, g_opt.reduce_tile_min.load(), 32)
                              : full;
    prm.tile_units = static_cast<int32_t>(tile);
    grid = plan_grid((prm.total_units + tile - 1) / tile, sms, occ);
  }
  return check_launch(launch_reduce(prm, dtype, order, grid, single, g_opt.pdl.load() != 0, stream),
                      what, single ? 1 : grid);
}

// Every reduction entry point: T tensors of P ranks; counts[t] is the
// element count per rank (all_reduce) or per shard (reduce_scatter).
dc_status_t reduce_entry(const void* const* in_ptrs, void* const* out_ptrs, const size_t* counts,
                         int T, int P, int dtype, int order, bool scatter, cudaStream_t stream,
                         const char* what) {
  read_env_once();
  if (P < 1 || P > kMaxRanks) return fail(DC_ERR_INVALID, "P = %d is outside 1..%d", P, kMaxRanks);
  if (dtype < kBF16 || dtype > kF32) return fail(DC_ERR_INVALID, "unknown element type %d", dtype);
  if (order != kOrderLinear && order != kOrderTree)
    return fail(DC_ERR_INVALID, "unknown summation order %d", order);
  if (T < 0) return fail(DC_ERR_INVALID, "T = %d is negative", T);
  const long long jobs = static_cast<long long>(T) * (scatter ? P : 1);
  if (jobs > kManyMaxReduceJobs || 2LL * T * P > kManyMaxReducePtrs)
    return fail(DC_ERR_TOO_MANY, "%d tensors x %d ranks exceed the %d jobs / %d pointers of one launch",
                T, P, kManyMaxReduceJobs, kManyMaxReducePtrs);
  if (T > 0 && !counts) return fail(DC_ERR_INVALID, "counts is NULL");
  std::vector<int> live;
  for (int t = 0; t < T; ++t)
    if (counts[t]) live.push_back(t);
  if (live.empty()) return ok();
  if (!in_ptrs || !out_ptrs) return fail(DC_ERR_INVALID, "in_ptrs and out_ptrs must not be NULL");
  const uint64_t es = static_cast<uint64_t>(esize_of(dtype));
  std::vector<Range> ranges;
  std::vector<uint64_t> shard_bytes(T, 0);
  uint64_t in_bytes_per_rank = 0;
  for (int t : live) {
    const uint64_t n = counts[t];
    if (n > UINT64_MAX / es / static_cast<uint64_t>(P))
      return fail(DC_ERR_INVALID, "count of tensor %d overflows", t);
    const uint64_t out_b = n * es, in_b = out_b * (scatter ? static_cast<uint64_t>(P) : 1);
    shard_bytes[t] = out_b;
    in_bytes_per_rank += in_b;
    for (int q = 0; q < P; ++q) {
      const void* pin = in_ptrs[static_cast<size_t>(t) * P + q];
      const void* pout = out_ptrs[static_cast<size_t>(t) * P + q];
      if (!pin || !pout)
        return fail(DC_ERR_INVALID, "pointer of tensor %d rank %d is NULL", t, q);
      const uint64_t i = reinterpret_cast<uint64_t>(pin), o = reinterpret_cast<uint64_t>(pout);
      if ((i | o) & (es - 1))
        return fail(DC_ERR_ALIGN, "tensor %d rank %d: %s pointers must be %d-byte aligned", t, q,
                    dtype_name(dtype), static_cast<int>(es));
      if (i + in_b < i || o + out_b < o)
        return fail(DC_ERR_INVALID, "buffer of tensor %d rank %d wraps around", t, q);
      ranges.push_back(Range{i, i + in_b, t, q, false});
      ranges.push_back(Range{o, o + out_b, t, q, true});
    }
  }
  dc_status_t st = check_reduce_overlaps(ranges, scatter, shard_bytes.data());
  if (st != DC_OK) return st;
  const int nz = static_cast<int>(live.size());
  const int njobs = nz * (scatter ? P : 1), nptr = 2 * nz * P;
  if (njobs == 1 && nptr <= 2 * kMaxRanks) {
    ReduceParams1 prm{};
    fill_reduce(prm, P, dtype, scatter, live, in_ptrs, out_ptrs, counts);
    return launch_reduce_plan(prm, 0, dtype, order, in_bytes_per_rank, stream, what);
  }
  if (njobs <= kMaxRanks && nptr <= 4 * kMaxRanks) {
    ReduceParamsS prm{};
    fill_reduce(prm, P, dtype, scatter, live, in_ptrs, out_ptrs, counts);
    return launch_reduce_plan(prm, 1, dtype, order, in_bytes_per_rank, stream, what);
  }
  static thread_local ReduceParamsL prm;  // 18 KB: keep it off the stack
  std::memset(&prm, 0, sizeof prm);
  fill_reduce(prm, P, dtype, scatter, live, in_ptrs, out_ptrs, counts);
  return launch_reduce_plan(prm, 2, dtype, order, in_bytes_per_rank, stream, what);
}

// One rank's share of a reduction: P inputs folded into one output,
// element i of the output from element in_offset + i of every input.
dc_status_t reduce_one_entry(const void* const* in_ptrs, int P, uint64_t in_offset, uint64_t count,
                             void* out, int dtype, int order, cudaStream_t stream) {
  read_env_once();
  if (P < 1 || P > kMaxRanks) return fail(DC_ERR_INVALID, "P = %d is outside 1..%d", P, kMaxRanks);
  if (dtype < kBF16 || dtype > kF32) return fail(DC_ERR_INVALID, "unknown element type %d", dtype);
  if (order != kOrderLinear && order != kOrderTree)
    return fail(DC_ERR_INVALID, "unknown summation order %d", order);
  if (count == 0) return ok();
  if (!in_ptrs || !out) return fail(DC_ERR_INVALID, "in_ptrs and out must not be NULL");
  const uint64_t es = static_cast<uint64_t>(esize_of(dtype));
  if (in_offset > UINT64_MAX / es || count > UINT64_MAX / es - in_offset)
    return fail(DC_ERR_INVALID, "in_offset + count overflows");
  const uint64_t o = reinterpret_cast<uint64_t>(out);
  const uint64_t out_b = count * es, skip = in_offset * es;
  if (o & (es - 1))
    return fail(DC_ERR_ALIGN, "out: %s pointers must be %d-byte aligned", dtype_name(dtype), static_cast<int>(es));
  if (o + out_b < o) return fail(DC_ERR_INVALID, "output wraps around the address space");
  std::vector<Range> ranges;
  ranges.push_back(Range{o, o + out_b, 0, 0, true});
  for (int q = 0; q < P; ++q) {
    const uint64_t i = reinterpret_cast<uint64_t>(in_ptrs[q]);
    if (!i) return fail(DC_ERR_INVALID, "in_ptrs[%d] is NULL", q);
    if (i & (es - 1))
      return fail(DC_ERR_ALIGN, "in_ptrs[%d]: %s pointers must be %d-byte aligned", q, dtype_name(dtype),
                  static_cast<int>(es));
    if (i + skip < i || i + skip + out_b < i + skip) return fail(DC_ERR_INVALID, "input %d wraps around", q);
    // the elements read: [in_q + skip, in_q + skip + out_b); the output may be
    // exactly that range of one input (in place)
    ranges.push_back(Range{i + skip, i + skip + out_b, 0, q, false});
  }
  const uint64_t zero = 0;
  dc_status_t st = check_reduce_overlaps(ranges, false, &zero);
  if (st != DC_OK) return st;
  ReduceParams1 prm{};
  prm.P = P;
  for (int q = 0; q < P; ++q) prm.ptr[q] = reinterpret_cast<uint64_t>(in_ptrs[q]);
  prm.ptr[P] = o;
  ReduceJob& J = prm.job[0];
  J.in0 = 0;
  J.out0 = static_cast<uint16_t>(P);
  J.nout = 1;
  J.in_off = in_offset;
  J.count = count;
  J.ufirst = 0;
  prm.njobs = 1;
  prm.total_units = classify_reduce_job(prm, J, P, dtype);
  return launch_reduce_plan(prm, 0, dtype, order, out_b, stream, "reduce");
}

// The launch shape of a fused all-gather: G chunk CTAs per rank (chunks of
// at least fused_chunk_min bytes, at most kFusedMaxChunks, and all P * G
// CTAs resident at once: the cooperative launch needs them together), and
// the gather step's TMA ring (fused_tma, fused_stages stages of
// fused_sub_bytes), whose shared memory decides how many CTAs fit an SM.
// Fills bytes, chunk, G, P, wait_ns, tma, stages and sub of fp.
dc_status_t plan_fused(FusedParams& fp, uint64_t B, int P, int sms) {
  fp.tma = g_opt.fused_tma.load() ? 1 : 0;
  fp.stages = static_cast<int32_t>(std::min(std::max(g_opt.fused_stages.load(), 1LL), 32LL));
  const long long sub = std::max(16LL, g_opt.fused_sub_bytes.load()) / 16 * 16;
  fp.sub = static_cast<uint32_t>(std::min(sub, static_cast<long long>(kFusedMaxSmem)));
  const size_t smem = fused_smem_bytes(fp.tma, fp.stages, fp.sub);
  if (smem > kFusedMaxSmem)
    return fail(DC_ERR_INVALID, "the fused TMA ring (%d stages of %u bytes) exceeds %zu bytes of shared memory",
                fp.stages, fp.sub, kFusedMaxSmem);
  const uint64_t resident = static_cast<uint64_t>(sms) * static_cast<uint64_t>(fused_ctas_per_sm(smem));
  if (resident < static_cast<uint64_t>(P))
    return fail(DC_ERR_INVALID, "%d ranks need %d CTAs resident at once; the GPU holds %llu", P, P,
                static_cast<unsigned long long>(resident));
  const uint64_t cmin = static_cast<uint64_t>(std::max(16LL, g_opt.fused_chunk_min.load()));
  uint64_t G = std::min<uint64_t>({(B + cmin - 1) / cmin, static_cast<uint64_t>(kFusedMaxChunks),
                                   resident / static_cast<uint64_t>(P)});
  G = std::max<uint64_t>(G, 1);
  const uint64_t chunk = ((B + G - 1) / G + 15) / 16 * 16;
  fp.bytes = B;
  fp.chunk = chunk;
  fp.G = static_cast<int32_t>((B + chunk - 1) / chunk);
  fp.P = P;
  fp.wait_ns = static_cast<uint64_t>(std::max(g_opt.wait_limit_ns.load(), 1000LL));
  return DC_OK;
}

}  // namespace

extern "C" {

dc_status_t dc_all_gather(const void* const* peer_ptrs, int P, size_t bytes_per_rank, void* out,
                          dc_stream_t stream) {
  read_env_once();
  if (P < 1 || P > kMaxRanks) return fail(DC_ERR_INVALID, "P = %d is outside 1..%d", P, kMaxRanks);
  if (bytes_per_rank == 0) return ok();
  if (!peer_ptrs) return fail(DC_ERR_INVALID, "peer_ptrs is NULL");
  if (!out) return fail(DC_ERR_INVALID, "out is NULL");
  const uint64_t B = bytes_per_rank;
  if (B > UINT64_MAX / static_cast<uint64_t>(P))
    return fail(DC_ERR_INVALID, "P * bytes_per_rank overflows");
  const uint64_t o = reinterpret_cast<uint64_t>(out);
  const uint64_t total = B * static_cast<uint64_t>(P);
  if (o + total < o) return fail(DC_ERR_INVALID, "output range wraps around the address space");
  for (int r = 0; r < P; ++r) {
    const uint64_t s = reinterpret_cast<uint64_t>(peer_ptrs[r]);
    if (!s) return fail(DC_ERR_INVALID, "peer_ptrs[%d] is NULL", r);
    if (s + B < s) return fail(DC_ERR_INVALID, "peer %d range wraps around", r);
    if (overlaps(o, total, s, B))
      return fail(DC_ERR_OVERLAP, "output overlaps the payload of rank %d", r);
  }
  GatherTensor t{o, B, peer_ptrs};
  const bool allow_flat = g_opt.force_generic.load() == 0;
  // 16-byte aligned and not sent to one CTA: the TMA-engine copy
  if (allow_flat && g_opt.gather_bulk.load() && tensor_aligned(t, P, true) &&
      total >= static_cast<uint64_t>(g_opt.bulk_min_bytes.load()) &&
      !use_single(total, g_opt.gather_single_max.load()))
    return launch_bulk_plan(t, P, total, static_cast<cudaStream_t>(stream));
  GatherParams1 prm{};
  fill_gather(prm, &t, 1, P, allow_flat);
  return launch_gather_plan(prm, 0, total, static_cast<cudaStream_t>(stream));
}

dc_status_t dc_all_gather_many(const void* const* peer_ptrs, const size_t* bytes_per_rank,
                               void* const* outs, int T, int P, dc_stream_t stream) {
  read_env_once();
  if (P < 1 || P > kMaxRanks) return fail(DC_ERR_INVALID, "P = %d is outside 1..%d", P, kMaxRanks);
  if (T < 0) return fail(DC_ERR_INVALID, "T = %d is negative", T);
  if (T > kManyMaxTensors)
    return fail(DC_ERR_TOO_MANY, "T = %d exceeds %d tensors per call", T, kManyMaxTensors);
  if (static_cast<long long>(T) * P > kManyMaxSegments)
    return fail(DC_ERR_TOO_MANY, "T * P = %lld exceeds %d segments per call",
                static_cast<long long>(T) * P, kManyMaxSegments);
  if (T == 0) return ok();
  if (!peer_ptrs || !bytes_per_rank || !outs)
    return fail(DC_ERR_INVALID, "peer_ptrs, bytes_per_rank and outs must not be NULL");
  GatherTensor ts[kManyMaxTensors];
  uint64_t out_total = 0;
  int live = 0;
  for (int t = 0; t < T; ++t) {
    const uint64_t B = bytes_per_rank[t];
    ts[t] = GatherTensor{reinterpret_cast<uint64_t>(outs[t]), B, peer_ptrs + static_cast<size_t>(t) * P};
    if (B == 0) continue;
    ++live;
    if (!outs[t]) return fail(DC_ERR_INVALID, "outs[%d] is NULL", t);
    if (B > UINT64_MAX / static_cast<uint64_t>(P))
      return fail(DC_ERR_INVALID, "P * bytes_per_rank[%d] overflows", t);
    const uint64_t tot = B * static_cast<uint64_t>(P);
    if (ts[t].out + tot < ts[t].out) return fail(DC_ERR_INVALID, "outs[%d] range wraps around", t);
    out_total += tot;
    for (int r = 0; r < P; ++r) {
      const uint64_t s = reinterpret_cast<uint64_t>(ts[t].peers[r]);
      if (!s) return fail(DC_ERR_INVALID, "peer_ptrs[%d] (tensor %d, rank %d) is NULL", t * P + r, t, r);
      if (s + B < s) return fail(DC_ERR_INVALID, "tensor %d rank %d range wraps around", t, r);
    }
  }
  if (live == 0) return ok();
  const dc_status_t ov = check_gather_overlaps(ts, T, P);
  if (ov != DC_OK) return ov;
  const bool allow_flat = g_opt.force_generic.load() == 0;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (live <= kManySmallTensors && live * P <= kManySmallSegments) {
    GatherParamsS prm{};
    GatherTensor packed[kManySmallTensors];
    int n = 0;
    for (int t = 0; t < T; ++t)
      if (ts[t].bytes) packed[n++] = ts[t];
    fill_gather(prm, packed, n, P, allow_flat);
    return launch_gather_plan(prm, 1, out_total, s);
  }
  static thread_local GatherParamsL prm;  // 18 KB: keep it off the stack
  std::memset(&prm, 0, sizeof prm);
  fill_gather(prm, ts, T, P, allow_flat);
  return launch_gather_plan(prm, 2, out_total, s);
}

dc_status_t dc_all_reduce_bf16(const void* const* in_ptrs, void* const* out_ptrs, int P,
                               size_t count, dc_stream_t stream) {
  return reduce_entry(in_ptrs, out_ptrs, &count, 1, P, kBF16, kOrderLinear, false,
                      static_cast<cudaStream_t>(stream), "all_reduce");
}

dc_status_t dc_reduce_scatter_bf16(const void* const* in_ptrs, void* const* out_ptrs, int P,
                                   size_t count_per_shard, dc_stream_t stream) {
  return reduce_entry(in_ptrs, out_ptrs, &count_per_shard, 1, P, kBF16, kOrderLinear, true,
                      static_cast<cudaStream_t>(stream), "reduce_scatter");
}

dc_status_t dc_all_reduce(const void* const* in_ptrs, void* const* out_ptrs, int P, size_t count,
                          dc_dtype_t dtype, dc_order_t order, dc_stream_t stream) {
  return reduce_entry(in_ptrs, out_ptrs, &count, 1, P, static_cast<int>(dtype),
                      static_cast<int>(order), false, static_cast<cudaStream_t>(stream), "all_reduce");
}

dc_status_t dc_reduce_scatter(const void* const* in_ptrs, void* const* out_ptrs, int P,
                              size_t count_per_shard, dc_dtype_t dtype, dc_order_t order,
                              dc_stream_t stream) {
  return reduce_entry(in_ptrs, out_ptrs, &count_per_shard, 1, P, static_cast<int>(dtype),
                      static_cast<int>(order), true, static_cast<cudaStream_t>(stream),
                      "reduce_scatter");
}

dc_status_t dc_reduce(const void* const* in_ptrs, int P, size_t in_offset, size_t count, void* out,
                      dc_dtype_t dtype, dc_order_t order, dc_stream_t stream) {
  return reduce_one_entry(in_ptrs, P, in_offset, count, out, static_cast<int>(dtype), static_cast<int>(order),
                          static_cast<cudaStream_t>(stream));
}

dc_status_t dc_all_reduce_many(const void* const* in_ptrs, void* const* out_ptrs,
                               const size_t* counts, int T, int P, dc_dtype_t dtype,
                               dc_order_t order, dc_stream_t stream) {
  return reduce_entry(in_ptrs, out_ptrs, counts, T, P, static_cast<int>(dtype),
                      static_cast<int>(order), false, static_cast<cudaStream_t>(stream),
                      "all_reduce_many");
}

dc_status_t dc_reduce_scatter_many(const void* const* in_ptrs, void* const* out_ptrs,
                                   const size_t* counts_per_shard, int T, int P, dc_dtype_t dtype,
                                   dc_order_t order, dc_stream_t stream) {
  return reduce_entry(in_ptrs, out_ptrs, counts_per_shard, T, P, static_cast<int>(dtype),
                      static_cast<int>(order), true, static_cast<cudaStream_t>(stream),
                      "reduce_scatter_many");
}

dc_status_t dc_inject_delay_ns(unsigned long long ns, dc_stream_t stream) {
  read_env_once();
  if (ns > DC_MAX_DELAY_NS)
    return fail(DC_ERR_INVALID, "delay %llu ns is above the %llu ns limit", ns,
                static_cast<unsigned long long>(DC_MAX_DELAY_NS));
  if (g_opt.test_fail_launch.load())
    return fail(DC_ERR_CUDA, "launch failure injected by the test_fail_launch option");
  return check_launch(launch_delay(ns, static_cast<cudaStream_t>(stream)), "delay", 1);
}

size_t dc_fused_workspace_bytes(int P) {
  return P < 1 || P > kMaxRanks ? 0 : fused_workspace_bytes(P);
}

dc_status_t dc_fused_all_gather(const void* const* in_ptrs, void* const* staging, void* const* outs, int P,
                                size_t bytes_per_rank, void* workspace, unsigned int epoch, dc_stream_t stream) {
  read_env_once();
  if (P < 1 || P > kMaxRanks) return fail(DC_ERR_INVALID, "P = %d is outside 1..%d", P, kMaxRanks);
  if (bytes_per_rank == 0) return ok();
  if (!in_ptrs || !staging || !outs) return fail(DC_ERR_INVALID, "in_ptrs, staging and outs must not be NULL");
  if (!workspace) return fail(DC_ERR_INVALID, "workspace is NULL");
  if (epoch == 0) return fail(DC_ERR_INVALID, "epoch 0 is reserved for a cleared workspace");
  const uint64_t B = bytes_per_rank;
  if (B > UINT64_MAX / static_cast<uint64_t>(P)) return fail(DC_ERR_INVALID, "P * bytes_per_rank overflows");
  const uint64_t total = B * static_cast<uint64_t>(P);
  const uint64_t ws = reinterpret_cast<uint64_t>(workspace), wsb = fused_workspace_bytes(P);
  if ((B & 15u) || (ws & 15u))
    return fail(DC_ERR_ALIGN, "bytes_per_rank and the workspace must be multiples of 16 bytes");
  // written ranges (staging buffers, outputs, workspace) may overlap nothing;
  // inputs may overlap each other
  struct R {
    uint64_t lo, hi;
    int kind, rank;  // kind 0 input, 1 staging, 2 output, 3 workspace
  };
  std::vector<R> v;
  v.reserve(3 * static_cast<size_t>(P) + 1);
  v.push_back(R{ws, ws + wsb, 3, 0});
  for (int r = 0; r < P; ++r) {
    const uint64_t a[3] = {reinterpret_cast<uint64_t>(in_ptrs[r]), reinterpret_cast<uint64_t>(staging[r]),
                           reinterpret_cast<uint64_t>(outs[r])};
    const uint64_t n[3] = {B, B, total};
    for (int k = 0; k < 3; ++k) {
      if (!a[k]) return fail(DC_ERR_INVALID, "a pointer of rank %d is NULL", r);
      if (a[k] & 15u) return fail(DC_ERR_ALIGN, "the buffers of rank %d must be 16-byte aligned", r);
      if (a[k] + n[k] < a[k]) return fail(DC_ERR_INVALID, "a buffer of rank %d wraps around", r);
      v.push_back(R{a[k], a[k] + n[k], k, r});
    }
  }
  std::sort(v.begin(), v.end(), [](const R& x, const R& y) { return x.lo < y.lo; });
  static const char* const kKind[4] = {"input", "staging buffer", "output", "workspace"};
  const R* far_any = nullptr;  // the range reaching furthest so far
  const R* far_w = nullptr;    // the written range reaching furthest so far
  for (const R& x : v) {
    const R* hit = x.kind == 0 ? far_w : far_any;
    if (hit && hit->hi > x.lo)
      return fail(DC_ERR_OVERLAP, "%s of rank %d overlaps %s of rank %d", kKind[x.kind], x.rank,
                  kKind[hit->kind], hit->rank);
    if (!far_any || x.hi > far_any->hi) far_any = &x;
    if (x.kind != 0 && (!far_w || x.hi > far_w->hi)) far_w = &x;
  }
  if (g_opt.test_fail_launch.load())
    return fail(DC_ERR_CUDA, "launch failure injected by the test_fail_launch option");
  int dev = 0, sms = 0;
  dc_status_t st = current_device(&dev);
  if (st != DC_OK) return st;
  st = sm_count(dev, &sms);
  if (st != DC_OK) return st;
  // G chunks per rank (one CTA each): chunks of at least fused_chunk_min
  // bytes, at most kFusedMaxChunks, and all P * G CTAs resident at once
  FusedParams fp{};
  st = plan_fused(fp, B, P, sms);
  if (st != DC_OK) return st;
  for (int r = 0; r < P; ++r) {
    fp.in[r] = reinterpret_cast<uint64_t>(in_ptrs[r]);
    fp.staging[r] = reinterpret_cast<uint64_t>(staging[r]);
    fp.out[r] = reinterpret_cast<uint64_t>(outs[r]);
  }
  fp.ws = ws;
  fp.absent = static_cast<uint64_t>(g_opt.test_fused_absent.load());
  fp.epoch = epoch;
  return check_launch(launch_fused_gather(fp, static_cast<cudaStream_t>(stream)), "fused all-gather",
                      P * fp.G);
}

dc_status_t dc_fused_all_gather_static(const void* const* in_ptrs, void* const* outs, int P,
                                       size_t bytes_per_rank, dc_stream_t stream) {
  read_env_once();
  if (P < 1 || P > kMaxRanks) return fail(DC_ERR_INVALID, "P = %d is outside 1..%d", P, kMaxRanks);
  if (bytes_per_rank == 0) return ok();
  if (!in_ptrs || !outs) return fail(DC_ERR_INVALID, "in_ptrs and outs must not be NULL");
  const uint64_t B = bytes_per_rank;
  if (B & 15u) return fail(DC_ERR_ALIGN, "bytes_per_rank must be a multiple of 16 bytes");
  if (B > kFusedStaticStagingBytes ||
      fused_static_stride(B) * static_cast<uint64_t>(P) > kFusedStaticStagingBytes)
    return fail(DC_ERR_INVALID,
                "%d ranks x %llu bytes need %llu bytes of staging; the static scratch holds %llu",
                P, static_cast<unsigned long long>(B),
                static_cast<unsigned long long>(fused_static_stride(std::min<uint64_t>(B, 1ull << 40)) * P),
                static_cast<unsigned long long>(kFusedStaticStagingBytes));
  const uint64_t total = B * static_cast<uint64_t>(P);
  // outputs may overlap nothing; inputs may overlap inputs
  struct R {
    uint64_t lo, hi;
    bool out;
    int rank;
  };
  std::vector<R> v;
  v.reserve(2 * static_cast<size_t>(P));
  for (int r = 0; r < P; ++r) {
    const uint64_t a = reinterpret_cast<uint64_t>(in_ptrs[r]), o = reinterpret_cast<uint64_t>(outs[r]);
    if (!a || !o) return fail(DC_ERR_INVALID, "a pointer of rank %d is NULL", r);
    if ((a | o) & 15u) return fail(DC_ERR_ALIGN, "the buffers of rank %d must be 16-byte aligned", r);
    if (a + B < a || o + total < o) return fail(DC_ERR_INVALID, "a buffer of rank %d wraps around", r);
    v.push_back(R{a, a + B, false, r});
    v.push_back(R{o, o + total, true, r});
  }
  std::sort(v.begin(), v.end(), [](const R& x, const R& y) { return x.lo < y.lo; });
  const R* far_any = nullptr;
  const R* far_out = nullptr;
  for (const R& x : v) {
    const R* hit = x.out ? far_any : far_out;
    if (hit && hit->hi > x.lo)
      return fail(DC_ERR_OVERLAP, "%s of rank %d overlaps %s of rank %d", x.out ? "output" : "input", x.rank,
                  hit->out ? "the output" : "the input", hit->rank);
    if (!far_any || x.hi > far_any->hi) far_any = &x;
    if (x.out && (!far_out || x.hi > far_out->hi)) far_out = &x;
  }
  if (g_opt.test_fail_launch.load())
    return fail(DC_ERR_CUDA, "launch failure injected by the test_fail_launch option");
  int dev = 0, sms = 0;
  dc_status_t st = current_device(&dev);
  if (st != DC_OK) return st;
  st = sm_count(dev, &sms);
  if (st != DC_OK) return st;
  FusedParams fp{};
  st = plan_fused(fp, B, P, sms);
  if (st != DC_OK) return st;
  for (int r = 0; r < P; ++r) {
    fp.in[r] = reinterpret_cast<uint64_t>(in_ptrs[r]);
    fp.out[r] = reinterpret_cast<uint64_t>(outs[r]);
  }
  fp.absent = 0;
  return check_launch(launch_fused_gather_static(fp, static_cast<cudaStream_t>(stream)),
                      "fused all-gather (static scratch)", P * fp.G);
}

dc_status_t dc_fused_reset(void* workspace, int P, dc_stream_t stream) {
  read_env_once();
  if (P < 1 || P > kMaxRanks) return fail(DC_ERR_INVALID, "P = %d is outside 1..%d", P, kMaxRanks);
  if (!workspace) return fail(DC_ERR_INVALID, "workspace is NULL");
  const cudaError_t e = cudaMemsetAsync(workspace, 0, fused_workspace_bytes(P), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DC_ERR_CUDA, "clearing the workspace failed: %s", cudaGetErrorString(e));
  }
  return ok();
}

dc_status_t dc_check_device(void) {
  read_env_once();
  uint32_t bits = 0, fused[4] = {0, 0, 0, 0};
  cudaError_t e = take_bulk_faults(&bits);
  if (e == cudaSuccess) e = take_fused_faults(fused);
  // bounds-check records of the checked build (empty in the normal build)
  static cudaError_t (*const kReaders[kBoundsReaders])(BoundsFault*) = {
      take_bounds_gather, take_bounds_bulk, take_bounds_fused,
      take_bounds_reduce_bf16, take_bounds_reduce_f16, take_bounds_reduce_f32};
  static const char* const kFiles[kBoundsReaders] = {"dc_gather.cu", "dc_bulk.cu", "dc_fused.cu",
                                                     "dc_reduce_bf16.cu", "dc_reduce_f16.cu", "dc_reduce_f32.cu"};
  BoundsFault first{};
  int first_file = -1;
  unsigned long long outside = 0;
  for (int i = 0; i < kBoundsReaders && e == cudaSuccess; ++i) {
    BoundsFault f{};
    e = kReaders[i](&f);
    if (e == cudaSuccess && f.count) {
      outside += f.count;
      if (first_file < 0) {
        first = f;
        first_file = i;
      }
    }
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(DC_ERR_CUDA, "device check failed: %s", cudaGetErrorString(e));
  }
  if (first_file >= 0)
    return fail(DC_ERR_BOUNDS,
                "%llu access(es) outside their job's range skipped; first: %s site %u, %llu bytes at 0x%llx, "
                "allowed [0x%llx, 0x%llx)",
                outside, kFiles[first_file], first.site, first.len, first.addr, first.lo, first.hi);
  if (fused[0] & kFaultFusedWait) {
    const uint32_t phase = fused[1] >> 24, rank = (fused[1] >> 12) & 0xFFFu, peer = fused[1] & 0xFFFu;
    return fail(DC_ERR_TIMEOUT,
                "fused all-gather: rank %u gave up waiting for rank %u's %s flag of chunk %u (epoch %u) "
                "after wait_limit_ns; clear the workspace (dc_fused_reset) and start again at epoch 1",
                rank, peer, phase == 1 ? "staged" : "done", fused[2], fused[3]);
  }
  if (bits & kFaultBulkWait)
    return fail(DC_ERR_TIMEOUT,
                "a bulk-copy all-gather gave up waiting for its loads after wait_limit_ns; "
                "its output is incomplete");
  return ok();
}

const char* dc_last_error(void) { return g_err; }

const char* dc_status_name(int status) {
  switch (status) {
    case DC_OK: return "DC_OK";
    case DC_ERR_INVALID: return "DC_ERR_INVALID";
    case DC_ERR_ALIGN: return "DC_ERR_ALIGN";
    case DC_ERR_OVERLAP: return "DC_ERR_OVERLAP";
    case DC_ERR_TOO_MANY: return "DC_ERR_TOO_MANY";
    case DC_ERR_CUDA: return "DC_ERR_CUDA";
    case DC_ERR_TIMEOUT: return "DC_ERR_TIMEOUT";
    case DC_ERR_BOUNDS: return "DC_ERR_BOUNDS";
    default: return "DC_ERR_UNKNOWN";
  }
}

int dc_set_option(const char* key, long long value) {
  read_env_once();
  if (!key || value < 0) return -1;
  for (const OptionKey& k : kKeys)
    if (std::strcmp(k.key, key) == 0) {
      k.slot->store(value);
      return 0;
    }
  return -1;
}

long long dc_get_option(const char* key) {
  read_env_once();
  if (!key) return -1;
  for (const OptionKey& k : kKeys)
    if (std::strcmp(k.key, key) == 0) return k.slot->load();
  return -1;
}

unsigned long long dc_launch_count(void) { return g_launches.load(); }

int dc_last_grid(void) { return g_last_grid; }

int dc_version(void) { return 1; }

int dc_bounds_checked(void) {
#ifdef DC_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

}  // extern "C"
