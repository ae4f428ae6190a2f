// Failure-detection self-test: a barrier wait that nothing completes must end
// by its time bound with W4A16_ETIMEOUT in the status word, leaving the
// context usable (no trap, no hang).  Uses the same bounded wait as the GEMM
// pipelines.
#include "common.cuh"
#include "kernels.h"

namespace w4a16 {

static __device__ int g_selftest_status;

__global__ void selftest_wait_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // phase 0 never completes: nobody arrives
        (void)mbar_wait(&bar, 0, &abort_flag, &g_selftest_status, limit_ns);
    }
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns);
    return cudaGetLastError();
}

int selftest_read_status() {
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_selftest_status, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    if (cudaMemcpyToSymbol(g_selftest_status, &zero, sizeof(int)) != cudaSuccess) return W4A16_ECUDA;
    return v;
}

}  // namespace w4a16
