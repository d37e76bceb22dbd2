// Test hook for the bounded waits of the TMA / tcgen05 kernels.
//
// Every mbarrier wait in those kernels gives up after a time limit, records
// an error bit in the handle's status word and lets the kernel return, so a
// missing arrival becomes an error status instead of a hung GPU.  This hook
// runs that same wait helper on an mbarrier that nothing ever arrives at,
// with a caller-chosen short limit, so a test can watch the wait run out and
// the status come back.
#include <cuda_runtime.h>

#include <cstdint>

#include "q4_tc.cuh"

namespace q4 {
namespace {

__global__ void wait_probe_kernel(int *status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = tc::smem_u32(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);                         // one arrival expected; none will come
        tc::mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait(b, 0, limit_ns)) atomicOr(status, 1);
}

}  // namespace

cudaError_t launch_wait_probe(int *status, uint64_t limit_ns, cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace q4
