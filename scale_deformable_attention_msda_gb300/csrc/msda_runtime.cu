// Host helpers: per-context addresses of the library's __device__ variables
// (the identity of a context comes from driver entry points reached through
// the runtime; the library does not link libcuda) and the device fault word of
// the range-checked build. Declared in msda_host.h.
#include <cudaTypedefs.h>

#include <mutex>

#include "msda_host.h"

namespace msda {

namespace {

// The device word per context that the checked build's kernels report into.
__device__ unsigned g_fault_word;

template <typename F>
F driver_entry(const char *name) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(fn);
}

struct DriverApi {
    PFN_cuCtxGetCurrent_v4000 ctx_get_current = nullptr;
    PFN_cuCtxGetId_v12000 ctx_get_id = nullptr;
};

const DriverApi &driver() {
    static DriverApi api;
    static std::once_flag once;
    std::call_once(once, [] {
        api.ctx_get_current = driver_entry<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent");
        api.ctx_get_id = driver_entry<PFN_cuCtxGetId_v12000>("cuCtxGetId");
    });
    return api;
}

// Identity of the calling thread's current context; false if there is none
// (yet) or the driver cannot tell.
bool current_context_id(unsigned long long *id) {
    const DriverApi &api = driver();
    if (!api.ctx_get_current || !api.ctx_get_id) return false;
    CUcontext ctx = nullptr;
    if (api.ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return api.ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

struct CachedAddress {
    const void *symbol;
    int device;
    unsigned long long ctx;
    void *address;
};
constexpr int kCacheSlots = 256;
std::mutex g_lock;
CachedAddress g_cache[kCacheSlots];
int g_used = 0;

}  // namespace

cudaError_t symbol_address(const void *symbol, void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    std::lock_guard<std::mutex> guard(g_lock);
    if (have_ctx) {
        for (int i = 0; i < g_used; ++i) {
            if (g_cache[i].symbol == symbol && g_cache[i].device == dev && g_cache[i].ctx == ctx) {
                *out = g_cache[i].address;
                return cudaSuccess;
            }
        }
    }
    // not cached for this context: look it up (this also creates the
    // primary context if none is current yet)
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    *out = p;
    unsigned long long now = 0;
    if (!current_context_id(&now)) return cudaSuccess;     // no identity: never cache
    for (int i = 0; i < g_used; ++i) {
        if (g_cache[i].symbol == symbol && g_cache[i].device == dev) {
            g_cache[i].ctx = now;                          // replaces the stale entry
            g_cache[i].address = p;
            return cudaSuccess;
        }
    }
    if (g_used < kCacheSlots) g_cache[g_used++] = CachedAddress{symbol, dev, now, p};
    return cudaSuccess;
}

cudaError_t fault_word(unsigned **out) {
    void *p = nullptr;
    const cudaError_t e = symbol_address(reinterpret_cast<const void *>(&g_fault_word), &p);
    *out = static_cast<unsigned *>(p);
    return e;
}

}  // namespace msda
