// noalloc.cu -- oscar_decode_attn_noalloc: decode attention for callers
// that cannot allocate device memory.
//
// oscar_decode_attn needs a caller-provided device workspace (rotated
// queries, the split-K plan and the split-K partials).  Some callers cannot
// provide one: code running where no allocator is reachable (inside a
// runtime that owns all device memory and hands out none, a plugin that may
// only use the buffers it is given), or code that must not allocate on a
// latency-critical path.  This entry point runs the same kernels with the
// workspace placed in a fixed-size array that lives in this library's own
// device image, so the call itself allocates nothing.
//
// In host code the array's name only stands in for the device object; its
// device address is looked up once per device with cudaGetSymbolAddress
// (with that device current) and passed to the kernels.
#include <mutex>

#include "oscar_common.cuh"

namespace oscar {

void set_last_cuda_error(int e);

namespace {

constexpr size_t kScratchBytes = OSCAR_NOALLOC_SCRATCH_BYTES;

// The scratch array.  Every GPU that loads this library's device code holds
// it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once).
cudaError_t scratch_on_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace oscar

extern "C" oscar_status oscar_decode_attn_noalloc(const oscar_shape* shape, int32_t batch, const void* q,
                                                  const void* bf16_kv, const int32_t* bf16_len, const uint8_t* pool,
                                                  const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                                                  const int32_t* hist_len, const float* U, float sm_scale,
                                                  float* out, int32_t* dev_status, void* stream) {
    // scratch this call would need; nothing is launched by the query
    size_t need = 0;
    oscar_status st = oscar_decode_attn(shape, batch, q, bf16_kv, bf16_len, pool, page_table, max_pages, num_pages,
                                        hist_len, U, sm_scale, out, nullptr, &need, dev_status, stream);
    if (st != OSCAR_OK) return st;
    if (need > oscar::kScratchBytes) return OSCAR_ERR_WORKSPACE;
    void* scratch = nullptr;
    const cudaError_t e = oscar::scratch_on_current_device(&scratch);
    if (e != cudaSuccess) {
        oscar::set_last_cuda_error((int)e);
        return OSCAR_ERR_CUDA;
    }
    // The kernels write every scratch word they later read (the plan and
    // the work counter are rebuilt at the start of each call), so nothing
    // left by an earlier call needs clearing.
    size_t have = oscar::kScratchBytes;
    return oscar_decode_attn(shape, batch, q, bf16_kv, bf16_len, pool, page_table, max_pages, num_pages, hist_len,
                             U, sm_scale, out, scratch, &have, dev_status, stream);
}
