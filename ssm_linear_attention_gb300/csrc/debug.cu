// debug.cu -- rssm_debug_pipeline_copy: a test of the streaming pipeline's bounded
// waits and its wind-down.
//
// The entry point copies n_tiles tiles of 16 KB from src to dst through the same
// warp-specialised pipeline (pipeline.cuh) the decode kernels use: the producer
// stages each tile with a 1-D bulk copy, the consumer warps write it out. With
// stall_tile >= 0 the producer arms that tile's stage for 16 bytes more than its copy
// delivers, so the stage's full barrier never completes although every issued copy
// lands. The consumer waiting for it gives up after wait_us microseconds, sets
// RSSM_DEVERR_TIMEOUT and the abort flag; the other warps of that CTA give up at once,
// and each producer waits (bounded) for the copies it issued before it exits. No copy
// is left in flight and no wait is unbounded, so the kernel returns and the context
// stays usable. The other CTAs copy their tiles normally.
#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace rssm {
namespace dbg {

constexpr int kTileBytes = 16384;
constexpr int kTileFloats = kTileBytes / 4;

struct CopyPolicy {
    static constexpr int kGroup = 2;
    struct Args {
        const float* src;
        float* dst;
        int32_t* dev_err;
        uint64_t wait_ns;
        int n, stall;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
    };
    struct Meta {
        int item;
    };

    static __device__ int n_items(const Args& a) { return a.n; }
    static __device__ int4 prefetch(const Args&, int) { return make_int4(0, 0, 0, 0); }

    static __device__ void issue(const Args& a, int item, int4, Meta* meta, uint8_t* sb,
                                 uint64_t* full, uint64_t pol) {
        meta->item = item;
        mbar_arrive_expect_tx(full, kTileBytes + (item == a.stall ? 16 : 0));
        bulk_g2s_hint(sb, a.src + (size_t)item * kTileFloats, kTileBytes, full, pol);
    }

    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb, uint8_t*,
                                   int lane, int wi) {
        const float4* s = reinterpret_cast<const float4*>(sb);
        float4* d = reinterpret_cast<float4*>(a.dst + (size_t)m.item * kTileFloats);
        constexpr int kVec = kTileFloats / 4 / kGroup;  // float4s per warp
        for (int i = lane; i < kVec; i += 32) d[wi * kVec + i] = s[wi * kVec + i];
    }
};

}  // namespace dbg
}  // namespace rssm

using namespace rssm;

extern "C" int rssm_debug_pipeline_copy(const float* src, float* dst, int n_tiles, int stall_tile,
                                        int wait_us, int32_t* dev_err, rssm_stream_t stream) {
    if (n_tiles < 0 || wait_us < 1 || wait_us > 2000000 || stall_tile >= n_tiles)
        return RSSM_ERR_INVALID_ARG;
    if (n_tiles == 0) return RSSM_OK;
    if (!ok_ptr(src) || !ok_ptr(dst)) return RSSM_ERR_INVALID_ARG;
    dbg::CopyPolicy::Args a{};
    a.src = src;
    a.dst = dst;
    a.dev_err = dev_err;
    a.wait_ns = (uint64_t)wait_us * 1000ull;
    a.n = n_tiles;
    a.stall = stall_tile < 0 ? -1 : stall_tile;
    return launch_pipe<dbg::CopyPolicy>(a, dbg::kTileBytes, 0, dbg::kTileBytes, n_tiles,
                                        (cudaStream_t)stream);
}
