/*
 * dc.h -- C ABI of libdc: the data-parallel core of a deterministic
 * collective on one GPU, with the world's P ranks held as P buffers in the
 * GPU's own memory.
 *
 * Pages cited by title:
 *   [PR491] "perf(cuda): vectorize the deterministic all-gather copy and
 *           right-size its single-block path" (RL-Kernel pull request 491).
 *
 * Conventions for every entry point:
 *   - Pointers named *_ptrs / outs / bytes_per_rank are HOST arrays that the
 *     call reads before it returns; the pointers stored in them are DEVICE
 *     addresses of the current device (cudaMalloc, torch CUDA tensors, or
 *     managed memory).  The caller owns all memory.
 *   - The work is enqueued on `stream` (NULL = the legacy default stream) and
 *     runs asynchronously.  A call allocates no memory, never synchronises,
 *     launches at most one kernel, and copies every pointer and size into the
 *     kernel's parameters, so it may be captured into a CUDA graph and the
 *     host arrays may be freed as soon as it returns.
 *   - Arguments are checked before any CUDA call; a rejected call launches
 *     nothing and returns a status with a message in dc_last_error().  A
 *     launch failure returns DC_ERR_CUDA.  Faults inside the kernel surface at
 *     the caller's next synchronisation, as for any CUDA kernel.
 *   - A call whose size is zero succeeds without launching anything (after P
 *     has been checked).
 *   - Results never depend on the path, grid size or stream timing: the
 *     gathers are exact byte copies and the reductions use one fixed
 *     per-element order.
 *   - Calls are thread-safe; options (dc_set_option) are process-wide.
 */
#ifndef DC_H
#define DC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *dc_stream_t;

typedef enum {
    DC_OK = 0,
    DC_ERR_INVALID = 1,  /* bad count, null pointer, size overflow */
    DC_ERR_ALIGN = 2,    /* a BF16 pointer that is not 2-byte aligned */
    DC_ERR_OVERLAP = 3,  /* an output range overlaps an input or another output */
    DC_ERR_TOO_MANY = 4, /* all_gather_many table larger than the limits below */
    DC_ERR_CUDA = 5,     /* the CUDA runtime refused the launch */
    DC_ERR_TIMEOUT = 6,  /* a bounded device wait ran out (reported by dc_check_device) */
    DC_ERR_BOUNDS = 7    /* bounds-checked build only: a kernel skipped an access outside its
                            job's range (reported by dc_check_device) */
} dc_status_t;

/* Element types and summation orders of the reductions. */
typedef enum { DC_BF16 = 0, DC_F16 = 1, DC_F32 = 2 } dc_dtype_t;
typedef enum { DC_ORDER_LINEAR = 0, DC_ORDER_TREE = 1 } dc_order_t;

#define DC_MAX_RANKS 64          /* P <= 64 */
#define DC_MANY_MAX_TENSORS 256  /* all_gather_many: T <= 256 */
#define DC_MANY_MAX_SEGMENTS 1024 /* all_gather_many: T * P <= 1024 */
#define DC_MANY_MAX_REDUCE_JOBS 256  /* reductions: T (all_reduce) or T * P (reduce_scatter) <= 256 */
#define DC_MANY_MAX_REDUCE_PTRS 1024 /* reductions: 2 * T * P <= 1024 */

/*
 * dc_all_gather -- rank-ordered all-gather ([PR491] section "What",
 * copy_rank_ordered bullet; the Python API there is all_gather(input, out=)).
 *
 *   out[r*bytes_per_rank + j] = peer_ptrs[r][j]   for r < P, j < bytes_per_rank.
 *
 * peer_ptrs: host array of P device pointers, each to bytes_per_rank bytes
 *            (any alignment; peers may overlap or repeat each other).
 * P:         1..DC_MAX_RANKS.
 * out:       device pointer to P*bytes_per_rank bytes, any alignment; it must
 *            not overlap any peer range (DC_ERR_OVERLAP).
 * Bytes outside [out, out + P*bytes_per_rank) are never written.
 * Path: the 16-byte flat vector copy when out, bytes_per_rank and every peer
 * are 16-byte aligned (staged through shared memory with cp.async, or, with
 * the gather_bulk option, bulk copies on the TMA engine); the realigning copy
 * otherwise (across the lanes of a warp, or through a shared-memory ring);
 * one CTA below the measured single-block threshold (output bytes), a grid
 * sized from the 16-byte vector count and the SM count above it.
 */
dc_status_t dc_all_gather(const void *const *peer_ptrs, int P, size_t bytes_per_rank,
                          void *out, dc_stream_t stream);

/*
 * dc_all_gather_many -- T independent all-gathers in one launch, each into
 * its own output, with no packing ([PR491] results paragraph and the
 * author's reply on all_gather_many: several gathers, one handshake, no
 * packing).
 *
 * peer_ptrs:      host array of T*P device pointers, tensor-major:
 *                 peer_ptrs[t*P + r] is rank r's payload of tensor t.
 * bytes_per_rank: host array of T sizes (zero allowed).
 * outs:           host array of T device pointers; outs[t] receives
 *                 P*bytes_per_rank[t] bytes in rank order.  Outputs must not
 *                 overlap each other or any payload.
 * T:              0..DC_MANY_MAX_TENSORS, and T*P <= DC_MANY_MAX_SEGMENTS
 *                 (DC_ERR_TOO_MANY otherwise).
 */
dc_status_t dc_all_gather_many(const void *const *peer_ptrs, const size_t *bytes_per_rank,
                               void *const *outs, int T, int P, dc_stream_t stream);

/*
 * dc_all_reduce_bf16 -- deterministic all_reduce of P BF16 buffers
 * ([PR491] sections "What" and "Not in this PR"; the page does not print the
 * arithmetic, and this is the reading used): for every i < count,
 *
 *   acc = f32(in_ptrs[0][i]);  acc = acc + f32(in_ptrs[q][i]) for q = 1..P-1
 *   (binary32, round to nearest even, in that order);
 *   out_ptrs[r][i] = bf16_round_nearest_even(acc) for every r < P.
 *
 * in_ptrs, out_ptrs: host arrays of P device pointers to `count` BF16
 *            elements each, 2-byte aligned (DC_ERR_ALIGN).  out_ptrs[r] may
 *            be exactly equal to an input pointer (in place); any other
 *            overlap between outputs and inputs, or between outputs, is
 *            DC_ERR_OVERLAP.  Inputs may overlap each other.
 * Subnormals are kept; NaN inputs give a NaN (payload unspecified).
 */
dc_status_t dc_all_reduce_bf16(const void *const *in_ptrs, void *const *out_ptrs, int P,
                               size_t count, dc_stream_t stream);

/*
 * dc_reduce_scatter_bf16 -- deterministic reduce_scatter: input = world x
 * output, as the author's reply on [PR491] describes it.  Each input holds
 * P*count_per_shard BF16 elements; rank r receives shard r:
 *
 *   out_ptrs[r][j] = fold over q = 0..P-1 of in_ptrs[q][r*count_per_shard + j]
 *
 * with the fold of dc_all_reduce_bf16.  out_ptrs[r] may be exactly
 * in_ptrs[q] + r*count_per_shard for some q (in place); other overlaps are
 * DC_ERR_OVERLAP.  Pointers must be 2-byte aligned.
 */
dc_status_t dc_reduce_scatter_bf16(const void *const *in_ptrs, void *const *out_ptrs, int P,
                                   size_t count_per_shard, dc_stream_t stream);

/*
 * dc_all_reduce / dc_reduce_scatter -- the same operations for any element
 * type and either summation order.  Every element is widened exactly to
 * binary32, the P values of an element are added one binary32 add (round to
 * nearest even) at a time in `order`, and the total is rounded once to
 * `dtype` (round to nearest even; DC_F32 totals are stored as they are):
 *   DC_ORDER_LINEAR: ((x0 + x1) + x2) + ... + x_{P-1};
 *   DC_ORDER_TREE:   fold(x[lo..hi)) = fold(x[lo..lo+m)) + fold(x[lo+m..hi)),
 *                    m the largest power of two below hi - lo.
 * [PR491] names a fixed-tree backend ("cuda_ipc_fixed_tree", author's
 * replies) without its shape; DC_ORDER_TREE is the plainest reading, and
 * DC_ORDER_LINEAR the default of the BF16 entry points above.  Pointers must
 * be aligned to the element size (2 or 4 bytes); aliasing rules as above.
 * Speed, not results, depends on alignment: the work runs in 16-byte units
 * anchored at the outputs when all outputs sit at the same address mod 16
 * (inputs at another offset are realigned, at about half the bandwidth), and
 * element by element otherwise.
 */
dc_status_t dc_all_reduce(const void *const *in_ptrs, void *const *out_ptrs, int P, size_t count,
                          dc_dtype_t dtype, dc_order_t order, dc_stream_t stream);
dc_status_t dc_reduce_scatter(const void *const *in_ptrs, void *const *out_ptrs, int P,
                              size_t count_per_shard, dc_dtype_t dtype, dc_order_t order,
                              dc_stream_t stream);

/*
 * dc_reduce -- one rank's share of a reduction: the P inputs folded into ONE
 * output, as dc_all_reduce / dc_reduce_scatter fold them:
 *
 *   out[i] = round(fold over q = 0..P-1 of in_ptrs[q][in_offset + i]),  i < count
 *
 * When every rank is its own process ([PR491] author's replies: the
 * collective's ranks exchange payloads through buffers their peers map),
 * rank r computes only its own output: its all_reduce output (in_offset 0,
 * count = elements per rank) or its reduce_scatter shard (in_offset =
 * r * count_per_shard, count = count_per_shard), from the P mapped buffers.
 * The result is bit-identical to the same rank's output of dc_all_reduce /
 * dc_reduce_scatter.
 *
 * in_ptrs: host array of P device pointers (read during the call), each to
 *          at least in_offset + count elements; aligned to the element size
 *          (DC_ERR_ALIGN).  Inputs may overlap each other.
 * out:     device pointer to count elements, aligned to the element size.
 *          It may be exactly the range of one input that is read (in_ptrs[q]
 *          + in_offset elements: in place); any other overlap with the
 *          elements read is DC_ERR_OVERLAP.
 * count:   0 is a successful no-op.  in_offset + count must not overflow
 *          (DC_ERR_INVALID).
 * One kernel on `stream`; nothing allocated, no synchronisation.
 */
dc_status_t dc_reduce(const void *const *in_ptrs, int P, size_t in_offset, size_t count, void *out,
                      dc_dtype_t dtype, dc_order_t order, dc_stream_t stream);

/*
 * dc_all_reduce_many / dc_reduce_scatter_many -- T independent reductions of
 * the same P, type and order in one launch ([PR491] "Tests":
 * reduce_scatter_many(..., outs=) with caller-given outputs).
 * in_ptrs, out_ptrs: host arrays of T*P device pointers, tensor-major
 *                    (tensor t, rank r at index t*P + r).
 * counts / counts_per_shard: host array of T element counts (zero allowed).
 * Limits: DC_MANY_MAX_REDUCE_JOBS jobs (T for all_reduce, T*P for
 * reduce_scatter) and 2*T*P <= DC_MANY_MAX_REDUCE_PTRS (DC_ERR_TOO_MANY).
 * Outputs may alias only their own tensor's inputs, as in the single forms.
 */
dc_status_t dc_all_reduce_many(const void *const *in_ptrs, void *const *out_ptrs,
                               const size_t *counts, int T, int P, dc_dtype_t dtype,
                               dc_order_t order, dc_stream_t stream);
dc_status_t dc_reduce_scatter_many(const void *const *in_ptrs, void *const *out_ptrs,
                                   const size_t *counts_per_shard, int T, int P, dc_dtype_t dtype,
                                   dc_order_t order, dc_stream_t stream);

/*
 * dc_inject_delay_ns -- keeps one GPU thread busy for `ns` nanoseconds of
 * the GPU's global timer, in stream order.  The rank-skew calibration
 * ("[Benchmark] Add all-reduce rank-skew calibration", vLLM pull request
 * 57037, section "Purpose") puts it on one simulated rank's stream before
 * that rank arrives at the collective.
 *
 * ns:     0..DC_MAX_DELAY_NS (DC_ERR_INVALID above); 0 launches a kernel
 *         that returns at once.
 * stream: the stream to delay.
 * The kernel reads no memory and writes none.  It stops when the timer has
 * advanced by ns, or, should the timer stall, after 4*ns + 2^20 SM cycles.
 * The requested delay is a lower bound on the kernel's duration; time it
 * with events to get the measured delay.
 */
#define DC_MAX_DELAY_NS 1000000000ull
dc_status_t dc_inject_delay_ns(unsigned long long ns, dc_stream_t stream);

/*
 * dc_fused_all_gather -- the staged all-gather protocol of the collective's
 * multi-rank deployment ([PR491] author's replies: the cuda_ipc_fixed_tree
 * backend's CUDA-graph-safe fused protocol, stage -> gather -> complete;
 * section "Not in this PR" and the review threads: a failed launch leaves the
 * protocol pending with no abort path, and peers of a dead rank wait for the
 * process-group timeout), run with the P ranks as CTA groups of one
 * cooperative launch on one GPU, every wait bounded.
 *
 * Rank r stages in_ptrs[r] into staging[r], publishes it, gathers every
 * rank's staging buffer into outs[r] in rank order, and completes once every
 * rank has read its staging buffer.  Afterwards, for every r:
 *
 *   outs[r][q*bytes_per_rank + j] = in_ptrs[q][j]   (q < P, j < bytes_per_rank)
 *
 * and staging[r] holds a copy of in_ptrs[r].
 *
 * in_ptrs, staging, outs: host arrays of P device pointers (16-byte aligned);
 *            each input and staging buffer holds bytes_per_rank bytes, each
 *            output P*bytes_per_rank.  Staging buffers, outputs and the
 *            workspace may overlap nothing; inputs may overlap inputs.
 * bytes_per_rank: a multiple of 16 (DC_ERR_ALIGN otherwise); 0 is a no-op.
 * workspace: device memory of dc_fused_workspace_bytes(P) bytes, 16-byte
 *            aligned, owned by the caller and zero before its first use
 *            (cudaMemset, or dc_fused_reset).  It holds the ranks' epoch flags.
 * epoch:     1 for the first call after the workspace was cleared, then one
 *            more for each call (never 0).  Calls on one workspace must not
 *            overlap on the GPU: issue them on one stream.
 * Every wait for a peer's flag is bounded by the "wait_limit_ns" option.  If
 * one runs out (a rank that never arrives), the waiting CTAs record the fault
 * and return, the outputs are incomplete, and dc_check_device returns
 * DC_ERR_TIMEOUT naming the waiting and the awaited rank; clear the workspace
 * with dc_fused_reset and start again at epoch 1.  P ranks need P*G CTAs
 * resident at once (G chunks per rank, at least one): DC_ERR_INVALID if the
 * GPU cannot hold P of them.
 */
size_t dc_fused_workspace_bytes(int P); /* 0 if P is outside 1..DC_MAX_RANKS */
dc_status_t dc_fused_all_gather(const void *const *in_ptrs, void *const *staging, void *const *outs, int P,
                                size_t bytes_per_rank, void *workspace, unsigned int epoch,
                                dc_stream_t stream);
/* Clears a fused workspace of P ranks on `stream` (cudaMemsetAsync); the next
 * call on it uses epoch 1. */
dc_status_t dc_fused_reset(void *workspace, int P, dc_stream_t stream);

/*
 * dc_fused_all_gather_static -- dc_fused_all_gather for callers that cannot
 * allocate device memory.  The pages describe no such entry point: it is this
 * library's own addition.  Some callers are given only their input and output
 * buffers and may not call cudaMalloc themselves: a plug-in run by a host
 * framework that owns every device allocation, code whose device memory was
 * planned once up front, or code that must not call cudaMalloc/cudaFree
 * because those can synchronise the device.  This form needs no workspace and
 * no staging buffers from them.
 *
 * It computes what dc_fused_all_gather computes (outs[r] = in_ptrs[0] ||
 * in_ptrs[1] || ... for every r; same argument rules for in_ptrs, outs, P and
 * bytes_per_rank), with the epoch flags and the P staging buffers in one
 * static device array of the library: 16 MiB of staging after 64 KiB of
 * flags, held by every GPU that loads the library until the process exits.
 * Limit: P * (bytes_per_rank rounded up to 256) <= 16 MiB; a larger call is
 * rejected with DC_ERR_INVALID before anything is launched.
 *
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.  Each call enqueues on `stream` a clear of the flags
 * (cudaMemsetAsync, 64 KiB at most) and one kernel.  The first call made with
 * a device current looks up the array's device address on that device
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call in the process uses the same array on a given GPU, which keeps
 * the last call's contents: calls whose work overlaps on the GPU (issued on
 * different streams, or from different host threads) race and corrupt each
 * other's results; issue them on one stream.  Waits are bounded as in
 * dc_fused_all_gather and reported by dc_check_device.
 */
dc_status_t dc_fused_all_gather_static(const void *const *in_ptrs, void *const *outs, int P,
                                       size_t bytes_per_rank, dc_stream_t stream);

/*
 * dc_check_device -- reports the faults that this library's kernels recorded
 * on the current device since the last check, and clears them.
 *
 * The bulk-copy gather (the "gather_bulk" path of dc_all_gather) waits for
 * its loads, and dc_fused_all_gather for its peers' flags, with a bound
 * (option "wait_limit_ns", default one second of the GPU's global timer).  A
 * wait that runs out does not hang the stream: the kernel records the fault
 * in a device word, waits with the same bound for its own copies in flight
 * and returns, leaving that call's output incomplete.  No correct bulk launch
 * on a working GPU ever runs out; a fused launch runs out when a rank never
 * arrives.
 *
 * Synchronous: it first waits for all work on the current device
 * (cudaDeviceSynchronize), then reads and clears the fault words.
 * Returns DC_OK if no wait ran out, DC_ERR_TIMEOUT if one did, DC_ERR_BOUNDS
 * (bounds-checked build only, see dc_bounds_checked) if a kernel skipped an
 * access outside its range, DC_ERR_CUDA if the synchronisation or the read
 * failed (the CUDA error in dc_last_error()).
 */
dc_status_t dc_check_device(void);

/* Message describing the last failed call on this thread ("" if none). */
const char *dc_last_error(void);

/* Name of a status code, e.g. "DC_ERR_OVERLAP". */
const char *dc_status_name(int status);

/*
 * Process-wide tuning and test options.  Keys:
 *   "force_path"              0 = automatic, 1 = single CTA, 2 = multi CTA
 *   "force_generic"           1 = never use the flat aligned gather path
 *   "gather_single_max_bytes" dc_all_gather on one CTA up to this many output
 *                             bytes (default 0: the grid was never slower on
 *                             GB300; an unaligned gather of fewer than 128
 *                             bytes per rank always runs on one CTA)
 *   "gather_many_single_max_bytes"
 *                             dc_all_gather_many on one CTA up to this many
 *                             output bytes in all (default 16384, measured)
 *   "reduce_single_max_bytes" single-CTA reductions up to this many input
 *                             bytes per rank (default 0: the grid was never
 *                             slower on GB300)
 *   "grid_ctas"               0 = automatic, else the multi-CTA grid size
 *   "pdl"                     1 (default) = launch with programmatic stream
 *                             serialization, so a kernel's launch overlaps the
 *                             end of the previous kernel in the stream (it still
 *                             waits for that kernel before touching memory)
 *   "gather_staged"           1 (default) = aligned gathers stage their loads
 *                             through shared memory with cp.async
 *   "gather_split_cost_pct"   all_gather_many with aligned and unaligned
 *                             tensors: cost of a realigned 16-byte vector in
 *                             percent of a staged aligned one, for splitting
 *                             the grid between the two (default 250, measured)
 *   "gather_split_cost_warp_pct" the same when the unaligned part (more than
 *                             16 tensors) realigns across warps (default 100,
 *                             measured)
 *   "prefetch"                tiles per CTA whose inputs are prefetched into
 *                             L2 before the kernel waits for the previous
 *                             kernel in the stream (dc_all_gather on its
 *                             aligned and staged realigning paths, and the
 *                             reductions; 0 = off; default 1)
 *   "gather_tile_min"         staged aligned gathers: the smallest tile (in
 *                             16-byte vectors) that an output too small for a
 *                             full tile per CTA is cut into, so that it is
 *                             spread evenly over the SMs (default 512, measured)
 *   "reduce_tile_min"         one-tensor all_reduce: the smallest tile (in
 *                             16-byte units) that a reduction too small for a
 *                             full tile per CTA is cut into (default 64,
 *                             measured)
 *   "reduce_staged"           1 (default) = an all_reduce of one tensor whose
 *                             inputs sit at other offsets (mod 16 bytes) than
 *                             its outputs, P = 2, 4 or 8, stages its input
 *                             blocks through shared memory; 0 = realign in
 *                             registers
 *   "gather_bulk"             1 (default) = a 16-byte aligned dc_all_gather
 *                             (out, bytes_per_rank and every peer) of at least
 *                             gather_bulk_min_bytes output bytes runs on the
 *                             TMA engine: 1-D bulk copies global -> shared ->
 *                             global through a ring of shared-memory stages
 *   "gather_bulk_min_bytes"   see gather_bulk (default 0)
 *   "bulk_chunk_bytes"        largest chunk one bulk stage moves (default 16384)
 *   "bulk_chunk_min"          smallest chunk an output too small for one
 *                             full chunk per CTA is cut into (default 2048)
 *   "bulk_stages"             ring stages per CTA (default 6, at most 32)
 *   "bulk_ctas_per_sm"        bulk CTAs per SM (default 2)
 *   "bulk_prefetch"           bulk CTAs prefetch their sources into L2 this
 *                             many chunks ahead of their loads (default 1; at
 *                             most 64 MB ahead over the grid; 0 when
 *                             "prefetch" is 0)
 *   "wait_limit_ns"           bound of one device wait (default 1000000000;
 *                             at least 1000)
 *   "test_bulk_short_tx"      1 = every bulk CTA's first wait runs out (tests
 *                             of dc_check_device)
 *   "gather_realign_warp"     1 (default) = a dc_all_gather whose payloads or
 *                             output are not 16-byte aligned (at least 128
 *                             bytes per rank, output under 4 GiB), and the
 *                             unaligned tensors of a dc_all_gather_many with
 *                             more than 16 of them, realign their vectors
 *                             across the lanes of a warp, in registers;
 *                             0 = through a shared-memory ring
 *   "fused_chunk_min"         dc_fused_all_gather: smallest chunk per CTA
 *                             (default 32768 bytes; measured, 8 ranks x 4 MiB:
 *                             75.8 us at 32 KiB, 81.9 us at 64 KiB)
 *   "fused_tma"               1 (default) = the protocol's gather step streams
 *                             the staged chunks through the TMA engine (one
 *                             thread per CTA, bulk loads and stores through a
 *                             shared-memory ring); 0 = every thread copies
 *                             16-byte vectors
 *   "fused_stages", "fused_sub_bytes"  that ring: stages (1..32, default 3) of
 *                             bytes each (a multiple of 16, default 32768)
 *   "test_fused_absent_ranks" bit r set: rank r of dc_fused_all_gather never
 *                             arrives (tests of its bounded waits)
 *   "test_fail_launch"        1 = report DC_ERR_CUDA instead of launching
 * Environment variables DC_FORCE_PATH, DC_FORCE_GENERIC,
 * DC_GATHER_SINGLE_MAX_BYTES, DC_GATHER_MANY_SINGLE_MAX_BYTES,
 * DC_REDUCE_SINGLE_MAX_BYTES, DC_GRID_CTAS, DC_PDL,
 * DC_GATHER_STAGED, DC_GATHER_SPLIT_COST_PCT, DC_GATHER_SPLIT_COST_WARP_PCT, DC_PREFETCH, DC_GATHER_TILE_MIN,
 * DC_REDUCE_TILE_MIN, DC_REDUCE_STAGED, DC_GATHER_BULK, DC_GATHER_BULK_MIN_BYTES,
 * DC_BULK_CHUNK_BYTES, DC_BULK_CHUNK_MIN, DC_BULK_STAGES, DC_BULK_CTAS_PER_SM,
 * DC_BULK_PREFETCH, DC_GATHER_REALIGN_WARP, DC_FUSED_CHUNK_MIN, DC_FUSED_TMA, DC_FUSED_STAGES,
 * DC_FUSED_SUB_BYTES and DC_WAIT_LIMIT_NS set the initial values (read once,
 * at the first call).
 * dc_set_option returns 0, or -1 for an unknown key or a negative value.
 * dc_get_option returns the value, or -1 for an unknown key.
 */
int dc_set_option(const char *key, long long value);
long long dc_get_option(const char *key);

/* Kernels launched by this library since it was loaded (all threads). */
unsigned long long dc_launch_count(void);

/* CTAs in the grid of the calling thread's last successful launch (0 before
 * the first): a diagnostic of the planner's grid choice. */
int dc_last_grid(void);

/* ABI version: 1. */
int dc_version(void);

/*
 * 1 in the bounds-checked build of the library (libdc_bounds.so, compiled
 * with DC_DEBUG_BOUNDS), 0 in the normal one.  In the checked build every
 * global load, store and L2 prefetch of every kernel is first checked against
 * the range its job allows -- for a load, the 16-byte-block hull of the
 * source bytes the job reads (realigning copies read whole aligned blocks
 * around an unaligned span); for a store, the exact output range.  An access
 * outside is skipped (never made) and the first one is recorded;
 * dc_check_device then returns DC_ERR_BOUNDS with the file, site, address and
 * allowed range.  The kernels never trap.  It is a test build: slower, and
 * otherwise the same results.
 */
int dc_bounds_checked(void);

#ifdef __cplusplus
}
#endif
#endif /* DC_H */
