// selftest.cu -- failure-detection self-test of the bounded waits.
//
// Every wait of the library's kernels (mbarrier phases, copy completions) is
// bounded by %globaltimer; when a bound runs out the kernel sets bit 8 of the
// sticky device error word and unwinds instead of hanging.  This kernel takes
// that path on purpose and harmlessly: one thread waits on an mbarrier phase
// that nothing completes, with a caller-chosen bound, then raises the bit and
// returns.  No fault, no trap, nothing left running.
#include "photon_common.cuh"

namespace photon {
namespace {

__global__ void __launch_bounds__(32) wait_probe_kernel(unsigned long long limit_ns,
                                                        uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);   // expects one arrival that never comes
  mbar_init_fence();
  const unsigned long long t0 = global_timer_ns();
  bool done = false;
  while (!done) {
    done = mbar_try_wait(&bar, 0);
    if (!done && global_timer_ns() - t0 > limit_ns) break;
  }
  if (!done) raise_error(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_wait_probe(unsigned long long limit_ns, uint32_t* err, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaGetLastError();
}

}  // namespace photon
