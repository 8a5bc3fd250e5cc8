// selftest.cu -- exercises the bounded-wait path every pipelined kernel relies on
// (kvfix_selftest_wait): a wait that nothing will end gives up after a cycle limit, sets
// the timeout flag in the device status word and returns, and the context stays usable.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace kvfix {

static __device__ unsigned int g_status_selftest;

unsigned read_status_selftest(cudaStream_t stream) {
    unsigned h = 0, zero = 0;
    cudaMemcpyFromSymbolAsync(&h, g_status_selftest, sizeof h, 0, cudaMemcpyDeviceToHost, stream);
    cudaMemcpyToSymbolAsync(g_status_selftest, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    cudaStreamSynchronize(stream);
    return h;
}

// One warp.  Lane 0 waits on an mbarrier whose phase never completes (expected arrivals: 1,
// none made) and on a flag nothing sets, each for at most `limit` cycles, with the same
// polling primitive the pipelines use; on expiry it records FLAG_TIMEOUT.
__global__ void selftest_wait_kernel(long long limit, const volatile int* flag) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x != 0) return;
    bool done = false;
    const long long t0 = clock64();
    while (!done && clock64() - t0 < limit) done = mbar_try_wait(&bar, 0u);
    bool seen = false;
    const long long t1 = clock64();
    while (!seen && flag && clock64() - t1 < limit) seen = *flag != 0;
    if (!done || (flag && !seen)) atomicOr(&g_status_selftest, FLAG_TIMEOUT);
}

cudaError_t launch_selftest_wait(long long limit_cycles, const int* flag, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(limit_cycles, flag);
    return cudaGetLastError();
}

}  // namespace kvfix
