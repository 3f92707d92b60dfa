// internal.h -- host-side helpers shared by the librssm entry points.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>  // CUtensorMap and its enums only: the driver is reached through the runtime
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

// Shape of a warp-specialised pipeline (pipeline.cuh): one CTA per SM with
// `groups` consumer groups of `group_warps` warps and one producer warp, `stages`
// shared-memory stages of `stage_bytes` (a multiple of `groups`), and
// `warp_scratch` bytes of private scratch per consumer warp. Chosen so that, with
// every group busy on one stage, the remaining stages keep at least 64 KB (and at
// least two tiles) of copies in flight; more groups are preferred.
struct PipeCfg {
    int stages;
    int groups;
    int smem_bytes;
    int stage_off;
    int scratch_off;
};
bool pick_pipe(const DeviceInfo& di, int stage_bytes, int warp_scratch, int tile_bytes, int header,
               int max_stages, int group_warps, int max_groups, PipeCfg* out, int align = 128);

// A 2-D tensor map over a row-major matrix of `rows` x `cols` elements of
// `elem_bytes` (2: bf16, 4: fp32) at `base` (16-byte aligned, rows of cols *
// elem_bytes bytes, a multiple of 16), copied in boxes of box_rows x (128 /
// elem_bytes) elements -- one 128-byte row segment per box row -- with the 128-byte
// shared-memory swizzle (16-byte chunk j of box row r lands at chunk j ^ (r % 8)).
// false when the driver offers no encoder or rejects the arguments.
bool make_tmap_rows128(CUtensorMap* out, const void* base, int elem_bytes, uint64_t rows,
                       uint64_t cols, uint32_t box_rows);

}  // namespace rssm
