// Test kernel: the INT2 decode's code operands on the tensor cores.  Each
// case is one warp and one mma.sync.m16n8k16 (f16 x f16 -> fp32, C = 0, as
// both of the decode's products; bf16 x bf16 for comparison on the slots
// whose bit pattern is also a bf16 subnormal):
// A is built from two 32-bit code words per lane with the library's own
// operand helpers (code_swap, code_pair_lo / code_pair_hi, exactly as the K and V
// products build them: bytes 0 and 2 of a word give k-pair (2tq, 2tq+1),
// bytes 1 and 3 give (2tq+8, 2tq+9), rows gID and gID+8 come from the two
// words), B is given as bf16 or f16 bit patterns.  The A registers and D are
// returned for the host to check against exact arithmetic (built and run by
// tests/test_gpu_tc_operands.py).
#include "../../bit_kv_cache_evict_gb300/csrc/oscar_common.cuh"

template <int SLOT>
__device__ __forceinline__ void operands(uint32_t w0, uint32_t w1, uint32_t (&a)[4]) {
    const uint32_t s0 = oscar::code_swap(w0), s1 = oscar::code_swap(w1);
    a[0] = oscar::code_pair_lo<SLOT>(w0, s0);
    a[1] = oscar::code_pair_lo<SLOT>(w1, s1);
    a[2] = oscar::code_pair_hi<SLOT>(w0, s0);
    a[3] = oscar::code_pair_hi<SLOT>(w1, s1);
}

// words [case][32][2]; bmat [case][16 k][8 n] bf16 / f16 bits; aregs
// [case][32][4]; d [case][16 rows][8 cols]
__global__ void tc_code_operands(int f16, const int* slot, const uint32_t* words, const uint16_t* bmat,
                                 uint32_t* aregs, float* d) {
    const int c = blockIdx.x, lane = threadIdx.x, gID = lane >> 2, tq = lane & 3;
    const uint32_t w0 = words[((size_t)c * 32 + lane) * 2], w1 = words[((size_t)c * 32 + lane) * 2 + 1];
    uint32_t a[4];
    switch (slot[c]) {
        case 0: operands<0>(w0, w1, a); break;
        case 1: operands<1>(w0, w1, a); break;
        case 2: operands<2>(w0, w1, a); break;
        default: operands<3>(w0, w1, a); break;
    }
    const uint16_t* b = bmat + (size_t)c * 128;
    const uint32_t b0 = (uint32_t)b[(2 * tq) * 8 + gID] | ((uint32_t)b[(2 * tq + 1) * 8 + gID] << 16);
    const uint32_t b1 = (uint32_t)b[(2 * tq + 8) * 8 + gID] | ((uint32_t)b[(2 * tq + 9) * 8 + gID] << 16);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (f16)
        oscar::mma_f16_16816(acc, a[0], a[1], a[2], a[3], b0, b1);
    else
        oscar::mma_bf16_16816(acc, a[0], a[1], a[2], a[3], b0, b1);
    for (int i = 0; i < 4; ++i) aregs[((size_t)c * 32 + lane) * 4 + i] = a[i];
    float* dc = d + (size_t)c * 128;
    dc[gID * 8 + 2 * tq] = acc[0];
    dc[gID * 8 + 2 * tq + 1] = acc[1];
    dc[(gID + 8) * 8 + 2 * tq] = acc[2];
    dc[(gID + 8) * 8 + 2 * tq + 1] = acc[3];
}

extern "C" int run_tc_code_operands(int ncases, int f16, const int* slot, const uint32_t* words,
                                    const uint16_t* bmat, uint32_t* aregs, float* d) {
    int* ds = nullptr;
    uint32_t *dw = nullptr, *da = nullptr;
    uint16_t* db = nullptr;
    float* dd = nullptr;
    const size_t nc = (size_t)ncases;
    int rc = 1;
    if (cudaMalloc(&ds, nc * sizeof(int)) == cudaSuccess && cudaMalloc(&dw, nc * 64 * 4) == cudaSuccess &&
        cudaMalloc(&db, nc * 128 * 2) == cudaSuccess && cudaMalloc(&da, nc * 128 * 4) == cudaSuccess &&
        cudaMalloc(&dd, nc * 128 * 4) == cudaSuccess) {
        cudaMemcpy(ds, slot, nc * sizeof(int), cudaMemcpyHostToDevice);
        cudaMemcpy(dw, words, nc * 64 * 4, cudaMemcpyHostToDevice);
        cudaMemcpy(db, bmat, nc * 128 * 2, cudaMemcpyHostToDevice);
        tc_code_operands<<<ncases, 32>>>(f16, ds, dw, db, da, dd);
        cudaError_t e = cudaDeviceSynchronize();
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e == cudaSuccess) {
            cudaMemcpy(aregs, da, nc * 128 * 4, cudaMemcpyDeviceToHost);
            cudaMemcpy(d, dd, nc * 128 * 4, cudaMemcpyDeviceToHost);
            rc = 0;
        } else {
            rc = 2;
        }
    }
    cudaFree(ds);
    cudaFree(dw);
    cudaFree(db);
    cudaFree(da);
    cudaFree(dd);
    return rc;
}
