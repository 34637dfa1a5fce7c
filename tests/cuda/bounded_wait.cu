// Test kernel: the library's bounded mbarrier wait on a barrier that nothing
// ever arrives on.  The wait must give up after its poll budget and report
// the timeout, leaving the context usable (built and run by
// tests/test_gpu_bounded_wait.py).
#include "../../bit_kv_cache_evict_gb300/csrc/oscar_common.cuh"

__global__ void wait_never(int* out, int polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        oscar::mbar_init(&bar, 1);
        oscar::fence_mbar_init();
    }
    __syncthreads();
    const bool done = oscar::mbar_wait_bounded(&bar, 0, polls);  // phase 0 never completes
    if (threadIdx.x == 0) out[blockIdx.x] = done ? 1 : 2;
}

extern "C" int run_wait_never(int polls, int blocks, int* results, float* ms) {
    int* d = nullptr;
    if (cudaMalloc(&d, sizeof(int) * blocks) != cudaSuccess) return 1;
    cudaMemset(d, 0, sizeof(int) * blocks);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a);
    wait_never<<<blocks, 32>>>(d, polls);
    cudaEventRecord(b);
    cudaError_t e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaGetLastError();
    cudaEventElapsedTime(ms, a, b);
    cudaMemcpy(results, d, sizeof(int) * blocks, cudaMemcpyDeviceToHost);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}
