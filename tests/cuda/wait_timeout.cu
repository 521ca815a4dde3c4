// Bounded-wait self-test.  One CTA waits, with the kernels' own bounded
// mbarrier wait and a short limit, on a barrier that no thread ever arrives at.
// The wait must give up, record DCP_ERR_TIMEOUT in the status word and let the
// kernel return; a second kernel then checks that the context is still usable.
// Nothing here faults, traps or spins without a bound.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dcp_device.cuh"
#include "dcp_sm100.cuh"

using namespace dcp::sm100;

namespace {

__global__ void wait_never_signalled(uint64_t limit_ns, int* status, unsigned long long* elapsed_ns,
                                     int* gave_up) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);   // phase 0 completes only after one arrival: none comes
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t t0 = globaltimer_ns();
  const bool done = mbar_wait(smem_u32(&bar), 0u, limit_ns);
  if (!done) {
    dcp::set_status(status, DCP_ERR_TIMEOUT);
    atomicAdd(gave_up, 1);
  }
  __syncthreads();
  if (threadIdx.x == 0) *elapsed_ns = globaltimer_ns() - t0;
}

__global__ void count_threads(int* counter) { atomicAdd(counter, 1); }

}  // namespace

// Returns 0, or 1000 + the CUDA error of the waiting kernel, or 2000 + the CUDA
// error of the follow-up kernel.
extern "C" int wait_timeout_probe(unsigned long long limit_ns, int threads, int* status,
                                  unsigned long long* elapsed_ns, int* gave_up, int* counter) {
  wait_never_signalled<<<1, threads>>>(limit_ns, status, elapsed_ns, gave_up);
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return 1000 + (int)e;
  count_threads<<<2, 64>>>(counter);
  e = cudaDeviceSynchronize();
  return e == cudaSuccess ? 0 : 2000 + (int)e;
}
