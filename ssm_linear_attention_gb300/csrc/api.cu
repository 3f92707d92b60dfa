// api.cu -- status strings, device facts, and the cursor kernel of librssm.
//
// The cursor kernel gives every decode row its ring write position and flush flag
// on the device, so a captured step needs no host metadata ([M2] "ReplaySSM:
// cache SSM inputs for faster Mamba2 standard decode", 实现拆解 item 3;
// [GDN] "GDN ReplaySSM decode (Part A of RFC 28511)", 实现拆解 item 2; [SPEC]
// "[GDN] Support ReplaySSM Ring Spec-Verify", 实现拆解 items 2 and 4; [FI]
// "[Mamba] Add FlashInfer ReplaySSM backend", 实现拆解 item 1).
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "cursor.cuh"
#include "internal.h"

namespace rssm {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
std::once_flag g_info_once[kMaxDevices];
bool g_info_ok[kMaxDevices];

struct SmemEntry {
    const void* kernel;
    int device;
    int bytes;
};
std::mutex g_smem_mu;
SmemEntry g_smem[512];
int g_smem_n = 0;
}  // namespace

bool device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    std::call_once(g_info_once[dev], [dev]() {
        DeviceInfo d{};
        bool ok = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) ==
                      cudaSuccess &&
                  cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                         dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.smem_per_sm,
                                         cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                         dev) == cudaSuccess;
        if (!ok) cudaGetLastError();
        g_info[dev] = d;
        g_info_ok[dev] = ok;
    });
    *out = g_info[dev];
    return g_info_ok[dev];
}

bool ensure_smem_limit(const void* kernel, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lk(g_smem_mu);
    for (int i = 0; i < g_smem_n; ++i)
        if (g_smem[i].kernel == kernel && g_smem[i].device == dev) {
            if (g_smem[i].bytes >= bytes) return true;
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
                cudaSuccess) {
                cudaGetLastError();
                return false;
            }
            g_smem[i].bytes = bytes;
            return true;
        }
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (g_smem_n < 512) g_smem[g_smem_n++] = SmemEntry{kernel, dev, bytes};
    return true;
}

bool pick_pipe(const DeviceInfo& di, int stage_bytes, int warp_scratch, int tile_bytes, int header,
               int max_stages, int group_warps, int max_groups, PipeCfg* out, int align) {
    const int budget = di.max_smem_optin;
    int want = (65536 + tile_bytes - 1) / tile_bytes;
    if (want < 2) want = 2;
    for (int ng = max_groups; ng >= 1; --ng) {
        const int scratch_off = header;
        const int stage_off = (scratch_off + ng * group_warps * warp_scratch + align - 1) / align * align;
        int stages = (budget - stage_off) / stage_bytes;
        if (stages > max_stages) stages = max_stages;
        stages -= stages % ng;  // each stage always belongs to the same group
        const bool ok = ng > 1 ? (stages - ng >= want) : (stages >= 2);
        if (ok) {
            out->stages = stages;
            out->groups = ng;
            out->stage_off = stage_off;
            out->scratch_off = scratch_off;
            out->smem_bytes = stage_off + stages * stage_bytes;
            return true;
        }
    }
    return false;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;
}  // namespace

bool make_tmap_rows128(CUtensorMap* out, const void* base, int elem_bytes, uint64_t rows,
                       uint64_t cols, uint32_t box_rows) {
    std::call_once(g_encode_once, []() {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(f);
        else
            cudaGetLastError();  // this lookup's own error
    });
    if (!g_encode || (elem_bytes != 2 && elem_bytes != 4)) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * (cuuint64_t)elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(out, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                2, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ----------------------------------------------------------------------------
// cursor kernel
// ----------------------------------------------------------------------------

__global__ void cursor_kernel(int mode, int32_t* __restrict__ slot_wp, int32_t* __restrict__ slot_base,
                              uint8_t* __restrict__ slot_flush, const int32_t* __restrict__ ci,
                              const uint8_t* __restrict__ force, const int32_t* __restrict__ acc,
                              int batch, int num_slots, int L, int T, int32_t* __restrict__ row_wp,
                              uint8_t* __restrict__ row_flush, int32_t* __restrict__ dev_err) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int s = ci[b];
    if (mode == RSSM_CURSOR_STANDARD) {
        standard_cursor(b, s, num_slots, L, slot_wp, force, row_wp, row_flush, dev_err);
        return;
    }
    if (s < 0) return;
    if (s >= num_slots) {
        set_dev_err(dev_err, RSSM_DEVERR_SLOT);
        return;
    }
    if (mode == RSSM_CURSOR_SPEC_COMMIT) {
        int cnt = slot_wp[s];
        int base = slot_base[s];
        const int a = acc[b];
        if (cnt < 0 || cnt > L || base < 0 || base >= L || a < 0 || a > T) {
            set_dev_err(dev_err, RSSM_DEVERR_CURSOR);
            return;
        }
        if (slot_flush[s]) {
            base = (base + cnt) % L;
            cnt = 0;
        }
        cnt += a;
        const int f = cnt + T > L;
        slot_wp[s] = cnt;
        slot_base[s] = base;
        slot_flush[s] = static_cast<uint8_t>(f);
        if (row_wp) row_wp[b] = cnt;
        if (row_flush) row_flush[b] = static_cast<uint8_t>(f);
    } else {  // RESET
        slot_wp[s] = 0;
        if (slot_base) slot_base[s] = 0;
        if (slot_flush) slot_flush[s] = 0;
    }
}

}  // namespace rssm

using namespace rssm;

extern "C" const char* rssm_status_string(int status) {
    switch (status) {
        case RSSM_OK: return "ok";
        case RSSM_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad enum or size)";
        case RSSM_ERR_UNSUPPORTED: return "unsupported shape or dtype (no kernel instance in the library)";
        case RSSM_ERR_CONFIG: return "inconsistent configuration";
        case RSSM_ERR_CUDA: return "CUDA launch error";
        default: return "unknown status";
    }
}

extern "C" int rssm_abi_version(void) { return RSSM_ABI_VERSION; }

extern "C" int rssm_advance_cursors(int mode, int32_t* slot_wp, int32_t* slot_base,
                                    uint8_t* slot_flush, const int32_t* cache_indices,
                                    const uint8_t* force_flush, const int32_t* num_accepted,
                                    int32_t batch, int32_t num_slots, int32_t L, int32_t T,
                                    int32_t* row_wp, uint8_t* row_flush, int32_t* dev_err,
                                    rssm_stream_t stream) {
    if (batch < 0 || num_slots < 0) return RSSM_ERR_INVALID_ARG;
    if (mode != RSSM_CURSOR_STANDARD && mode != RSSM_CURSOR_SPEC_COMMIT && mode != RSSM_CURSOR_RESET)
        return RSSM_ERR_INVALID_ARG;
    if (L < 1) return RSSM_ERR_CONFIG;
    if (batch == 0) return RSSM_OK;
    if (!slot_wp || !cache_indices) return RSSM_ERR_INVALID_ARG;
    if (mode == RSSM_CURSOR_STANDARD && (!row_wp || !row_flush)) return RSSM_ERR_INVALID_ARG;
    if (mode == RSSM_CURSOR_SPEC_COMMIT) {
        if (!slot_base || !slot_flush || !num_accepted) return RSSM_ERR_INVALID_ARG;
        if (T < 1 || L < 2 * T) return RSSM_ERR_CONFIG;
    }
    const int threads = 256;
    cursor_kernel<<<(batch + threads - 1) / threads, threads, 0, (cudaStream_t)stream>>>(
        mode, slot_wp, slot_base, slot_flush, cache_indices, force_flush, num_accepted, batch,
        num_slots, L, T, row_wp, row_flush, dev_err);
    return launch_status();
}
