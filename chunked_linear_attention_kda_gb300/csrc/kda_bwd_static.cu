// kda_bwd_static.cu -- a fixed device scratch array for the backward pass's checkpoints,
// used by kda_chunk_bwd_static_scratch (an entry point that takes no workspace and makes
// no allocation). The array is static device memory of the loaded module: it exists once
// per device, for the lifetime of the library, shared by every call on that device.
#include <mutex>

#include "kda_internal.h"

namespace kda {
namespace {

__device__ __align__(256) unsigned char g_bwd_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_lock;
void *g_scratch_ptr[kMaxDevices];  // device address of g_bwd_scratch, looked up once per device

}  // namespace

cudaError_t static_scratch(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_lock);
    if (!g_scratch_ptr[dev]) {
        e = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_bwd_scratch);
        if (e != cudaSuccess) return e;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace kda
