// Self-test of the failure path: a bounded mbarrier wait that cannot complete.
//
// Every kernel of the library bounds its waits: when a wait runs out, the kernel
// sets a bit of the device error word (read and cleared by w4_device_error)
// and returns instead of hanging, so the context stays usable. This kernel
// exercises that path on purpose: its barrier expects one arrival that no
// thread makes, so the wait gives up after `limit` tests of at most ~20 us each.
#include "common.cuh"
#include "internal.h"

namespace w4 {

namespace {

__global__ void bounded_wait_selftest_kernel(int *err, int limit)
{
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_bounded(smem_addr(&bar), 0, limit))
        atomicOr(err, 4);
}

} // namespace

cudaError_t run_bounded_wait_selftest(int *err, cudaStream_t s)
{
    bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(err, 50); // gives up within ~1 ms
    return cudaGetLastError();
}

} // namespace w4
