// moe_clock_probe: samples the SM clock while other work runs, so that a measured
// rate can be compared with a peak taken at another clock.  One thread of one CTA
// records (%globaltimer, clock64) pairs every interval_ns for n samples; run on a
// stream of its own it shares an SM with whatever else is resident and sleeps
// between samples.  The pages have no counterpart: this is a measurement aid.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__global__ void clock_probe_kernel(uint64_t *__restrict__ samples, int n, uint64_t interval_ns) {
  if (threadIdx.x != 0) return;
  const uint64_t t0 = global_ns();
  for (int i = 0; i < n; ++i) {
    const uint64_t target = t0 + (uint64_t)i * interval_ns;  // the last target is t0 + (n - 1) interval_ns
    uint64_t t = global_ns();
    while (t < target) {
      __nanosleep(1000);
      t = global_ns();
    }
    samples[2 * i] = t;
    samples[2 * i + 1] = (uint64_t)clock64();
  }
}

}  // namespace
}  // namespace moe

extern "C" MOE_API int moe_clock_probe(uint64_t *samples, int n, int64_t interval_ns, void *stream) {
  using namespace moe;
  if (!samples || (reinterpret_cast<uintptr_t>(samples) & 7) || n < 2 || n > (1 << 20) || interval_ns < 1000 ||
      (int64_t)(n - 1) * interval_ns > 10000000000ll)
    return MOE_ERR_INVALID_ARG;
  // The SM hosting the probe must keep its whole shared memory available to the kernels
  // it shares the SM with: a probe resident under a small-shared-memory carveout
  // would keep a 200 KB CTA of another kernel off its SM until the probe ends.
  if (cudaFuncSetAttribute(clock_probe_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return MOE_ERR_CUDA;
  clock_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(samples, n, (uint64_t)interval_ns);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
