// mla_static_scratch.cu -- a fixed scratch region in the library's own device
// memory, used by mla_decode_forward_static (the forward pass for callers
// that provide no scratch buffer and must not allocate).  Host code plus one
// file-scope device array; nothing here allocates or frees.
#include <mutex>

#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "mla_internal.h"

// Zero-initialised when the module is loaded in a context; one copy per
// context (so per device, for the runtime's primary contexts).
static __device__ __align__(256) unsigned char g_static_scratch[mla::kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

// The array's address is a property of the context the module was loaded
// in: after a device reset (or any other end of the primary context) the
// module is loaded again, possibly at another address.  So the address is
// kept together with the id of the context it was looked up in, and a call
// made in another context looks it up again.
struct Entry {
    unsigned long long ctx_id = 0;   // 0: not looked up yet
    void* addr = nullptr;
};
Entry g_entries[kMaxDevices];
std::mutex g_static_mutex;

PFN_cuCtxGetCurrent_v4000 g_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_get_id = nullptr;
std::once_flag g_entry_points_once;

void load_entry_points() {
    std::call_once(g_entry_points_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult qr{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            g_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        else
            cudaGetLastError();
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            g_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
        else
            cudaGetLastError();
    });
}

// Id of the calling thread's current context; 0 if there is none (or the
// driver cannot say).
unsigned long long current_context_id() {
    load_entry_points();
    if (!g_get_current || !g_get_id) return 0;
    CUcontext ctx = nullptr;
    if (g_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (g_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace

namespace mla {

void* static_scratch_if_ready(int device) {
    if (device < 0 || device >= kMaxDevices) return nullptr;
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(g_static_mutex);
    const Entry& e = g_entries[device];
    if (id == 0 || e.ctx_id != id) return nullptr;
    return e.addr;
}

cudaError_t static_scratch_set_up(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    // The symbol's address in the current context (the caller made `device`
    // current; the lookup also creates the primary context if needed).
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e;
    }
    // id 0 (no context id available): nothing is cached, every call looks up
    Entry& en = g_entries[device];
    en.ctx_id = current_context_id();
    en.addr = p;
    *out = p;
    return cudaSuccess;
}

}  // namespace mla
