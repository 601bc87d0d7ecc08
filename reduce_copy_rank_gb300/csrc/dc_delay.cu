// Injected GPU delay for the rank-skew calibration.
//
// Page, by title: "[Benchmark] Add all-reduce rank-skew calibration" (vLLM
// pull request 57037), section "Purpose": one rank is delayed on the GPU
// before the collective, and the delay actually obtained is measured beside
// the requested one (the review's second suggestion: a delay converted to
// cycles with the rated clock drifts from the request, most at small delays).
//
// Here the delay is counted on the GPU's global nanosecond timer, so it does
// not depend on the SM clock.  The loop has a second stop, on the SM's cycle
// counter at four cycles per requested nanosecond plus 2^20 cycles (the SM
// clock is at most ~2.1 GHz, so this bound is never reached before the timer
// one while the timer runs): the kernel ends even if the timer stalls.  One
// thread, no memory access.
#include "dc_internal.h"

namespace dc {
namespace {

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void dc_delay_kernel(unsigned long long ns, unsigned long long max_cycles) {
  const unsigned long long t0 = global_ns();
  const long long c0 = clock64();
  while (global_ns() - t0 < ns) {
    if (static_cast<unsigned long long>(clock64() - c0) > max_cycles) break;
  }
}

}  // namespace

cudaError_t launch_delay(unsigned long long ns, cudaStream_t s) {
  const unsigned long long max_cycles = 4ull * ns + (1ull << 20);
  dc_delay_kernel<<<1, 1, 0, s>>>(ns, max_cycles);
  return cudaGetLastError();
}

}  // namespace dc
