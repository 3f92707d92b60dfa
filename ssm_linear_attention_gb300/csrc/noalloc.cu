// noalloc.cu -- rssm_mamba2_decode_noalloc: the Mamba2 ReplaySSM decode for callers
// that cannot allocate device memory.
//
// rssm_mamba2_decode needs a caller-provided workspace for its per-(row, head)
// coefficient tables. Some callers have no way to provide one: a plug-in running
// inside a host application that owns every device allocation, an engine whose
// device memory budget is fixed at start-up, or a caller on a latency-critical
// path that must never enter the allocator. This entry point keeps that workspace
// in a fixed array that lives in the library's own device image instead, so the
// caller passes only inputs and outputs and nothing is allocated per call.
//
// The array (RSSM_NOALLOC_WORKSPACE_BYTES) is part of the module: every GPU that
// loads the library holds it until the process exits. Every call on a device
// shares it and it keeps the previous call's contents; nothing in it needs to start
// at zero (each call writes the table rows it reads). Calls whose executions
// overlap on the GPU race on the array, so issue them in one stream or order them.
#include <mutex>

#include "internal.h"
#include "rssm.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_workspace[RSSM_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// The array's device address per device, with the id of the context it was looked
// up in. A device reset destroys that context and unloads the module, so a cached
// address is reused only while the device's current context is still the same one.
struct Cached {
    bool valid;
    unsigned long long ctx_id;
    void* ptr;
};
std::mutex g_mu;
Cached g_cache[kMaxDevices];

// Driver entry points (looked up through the runtime, so the library keeps loading on
// machines without a driver): the current context and its unique id.
typedef int (*CtxGetCurrentFn)(void**);
typedef int (*CtxGetIdFn)(void*, unsigned long long*);
std::once_flag g_drv_once;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

// Id of the calling thread's current context; false when there is none yet (the
// runtime creates it on first use) or the driver offers no such query.
bool current_context_id(unsigned long long* id) {
    std::call_once(g_drv_once, []() {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f);
        else
            cudaGetLastError();  // this lookup's own error
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<CtxGetIdFn>(f);
        else
            cudaGetLastError();
    });
    if (!g_ctx_current || !g_ctx_id) return false;
    void* ctx = nullptr;
    if (g_ctx_current(&ctx) != 0 || ctx == nullptr) return false;
    return g_ctx_id(ctx, id) == 0;
}

// Device address of the array for the current device. Host code must not use the
// symbol itself as a pointer: it names a host-side stand-in. The address is looked
// up with the device current, cached only when the look-up succeeds (a failed one,
// for instance inside a stream capture that forbids it, is retried by the next
// call), and looked up again when the device's context has changed since.
void* workspace_address(int* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();  // the error this call raised
        *status = RSSM_ERR_CUDA;
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *status = RSSM_ERR_UNSUPPORTED;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    Cached& c = g_cache[dev];
    if (c.valid && have_id && c.ctx_id == id) {
        *status = RSSM_OK;
        return c.ptr;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || p == nullptr) {
        cudaGetLastError();  // the error this call raised
        c.valid = false;
        *status = RSSM_ERR_CUDA;
        return nullptr;
    }
    // the look-up made the context current if there was none: take its id now
    c.valid = current_context_id(&c.ctx_id);
    c.ptr = p;
    *status = RSSM_OK;
    return p;
}

}  // namespace

extern "C" int rssm_mamba2_decode_noalloc(const rssm_mamba2_dims* d, void* state, const float* A,
                                          const void* C, const float* D, const void* z,
                                          const void* ring_x, const float* ring_dt,
                                          const void* ring_B, const int32_t* cache_indices,
                                          const int32_t* row_wp, const uint8_t* row_flush, void* y,
                                          int32_t* dev_err, rssm_stream_t stream) {
    if (!d) return RSSM_ERR_INVALID_ARG;
    const size_t need = rssm_mamba2_workspace_size(d);
    if (need == 0) {
        // invalid dims (or an empty batch): let the regular entry point report it
        return rssm_mamba2_decode(d, state, A, C, D, z, ring_x, ring_dt, ring_B, cache_indices,
                                  row_wp, row_flush, nullptr, 0, y, dev_err, stream);
    }
    if (need > (size_t)RSSM_NOALLOC_WORKSPACE_BYTES) return RSSM_ERR_UNSUPPORTED;
    int status = RSSM_OK;
    void* ws = workspace_address(&status);
    if (!ws) return status;
    return rssm_mamba2_decode(d, state, A, C, D, z, ring_x, ring_dt, ring_B, cache_indices, row_wp,
                              row_flush, ws, (size_t)RSSM_NOALLOC_WORKSPACE_BYTES, y, dev_err,
                              stream);
}
