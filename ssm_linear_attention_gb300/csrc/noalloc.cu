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
std::once_flag g_once[kMaxDevices];
void* g_ptr[kMaxDevices];
cudaError_t g_err[kMaxDevices];

// Device address of the array for the current device, looked up once per device
// with that device current. Host code must not use the symbol itself as a pointer.
void* workspace_address(int* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        *status = RSSM_ERR_CUDA;
        return nullptr;
    }
    std::call_once(g_once[dev], [dev]() {
        void* p = nullptr;
        g_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_workspace);
        if (g_err[dev] != cudaSuccess) cudaGetLastError();
        g_ptr[dev] = p;
    });
    if (g_err[dev] != cudaSuccess || g_ptr[dev] == nullptr) {
        *status = RSSM_ERR_CUDA;
        return nullptr;
    }
    *status = RSSM_OK;
    return g_ptr[dev];
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
