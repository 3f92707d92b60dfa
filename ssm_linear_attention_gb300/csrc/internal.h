// internal.h -- host-side helpers shared by the librssm entry points.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "rssm.h"

namespace rssm {

// Per-device launch facts, queried once per device.
struct DeviceInfo {
    int sm_count;
    int max_smem_optin;  // bytes per block
    int smem_per_sm;     // bytes per multiprocessor
};

// Facts for the current device; false if the runtime reports no device.
bool device_info(DeviceInfo* out);

// Raise a kernel's dynamic shared memory limit once per (kernel, device).
bool ensure_smem_limit(const void* kernel, int bytes);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
inline bool ok_opt_ptr(const void* p) { return p == nullptr || aligned16(p); }
inline bool ok_dtype(int d) { return d == RSSM_F32 || d == RSSM_BF16; }
inline int dtype_bytes(int d) { return d == RSSM_BF16 ? 2 : 4; }

inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

// Pick a persistent-grid shape for a streaming kernel with `stage_bytes` per
// pipeline stage plus `fixed_bytes` of other shared memory: prefer two resident
// CTAs per SM with >= 3 stages each, else one CTA with >= 2 stages.
struct PipeShape {
    int stages;
    int ctas_per_sm;
    int smem_bytes;
};
bool pick_pipe_shape(const DeviceInfo& di, int stage_bytes, int fixed_bytes, int max_stages,
                     PipeShape* out);

}  // namespace rssm
