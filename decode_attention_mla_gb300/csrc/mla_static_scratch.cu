// mla_static_scratch.cu -- a fixed scratch region in the library's own device
// memory, used by mla_decode_forward_static (the forward pass for callers
// that provide no scratch buffer and must not allocate).  Host code plus one
// file-scope device array; nothing here allocates or frees.
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "mla_internal.h"

// Zero-initialised when the module is loaded on a device; one copy per device.
static __device__ __align__(256) unsigned char g_static_scratch[mla::kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<void*> g_static_addr[kMaxDevices];
std::mutex g_static_mutex;

}  // namespace

namespace mla {

void* static_scratch_if_ready(int device) {
    if (device < 0 || device >= kMaxDevices) return nullptr;
    return g_static_addr[device].load(std::memory_order_acquire);
}

cudaError_t static_scratch_set_up(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    void* p = g_static_addr[device].load(std::memory_order_relaxed);
    if (!p) {
        // The symbol's address on the current device: the caller made `device` current.
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return e;
        }
        g_static_addr[device].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace mla
