// static_scratch.cu -- ds_sparse_attn_static_scratch: sparse_attn for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention: code that runs
// inside a custom memory manager or a runtime that owns every allocation, plugins that are
// handed only input and output buffers, and hosts that forbid allocation on their hot path.
// For them this file keeps the scratch that sparse_attn needs for tokens split across CTAs in a
// fixed device array compiled into the library, so the call needs nothing beyond its inputs and
// outputs.  Every device that loads the library reserves the array until the process exits.
#include <mutex>

#include "common.cuh"

namespace dsattn {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)32 << 20;   // 32 MiB

// The scratch itself.  In host code this name is only a stand-in for the device symbol, never an
// address a kernel may be given; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices];

// Device address of this device's copy of the scratch, looked up once per device with that
// device current.
void *static_scratch_for_current_device(int *status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = DS_ECUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
            *status = DS_ECUDA;
            return nullptr;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *status = DS_OK;
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace dsattn

extern "C" {

size_t ds_sparse_attn_static_scratch_capacity(void) { return dsattn::kStaticScratchBytes; }

int ds_sparse_attn_static_scratch(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink,
                                  const int32_t *idx, int topk, float scale, uint16_t *o, int b, int m, int h,
                                  int d, ds_stream_t stream) {
    int status = DS_OK;
    void *scratch = dsattn::static_scratch_for_current_device(&status);
    if (!scratch) return status;
    // Same checks, kernels and results as ds_sparse_attn; a shape whose scratch need exceeds the
    // static array is refused there with DS_EWORKSPACE before anything is launched.
    return ds_sparse_attn(q, kv, n, sink, idx, topk, scale, o, b, m, h, d, scratch, dsattn::kStaticScratchBytes,
                          stream);
}

}  // extern "C"
