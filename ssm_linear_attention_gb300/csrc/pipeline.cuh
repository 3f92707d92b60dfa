// pipeline.cuh -- persistent, warp-specialised streaming pipeline for sm_103a.
//
// One CTA per SM holds `groups` independent pipelines. Each pipeline has one
// producer warp and one consumer group of K::kGroup warps:
//   * the producer's lanes prefetch the row metadata of its next 32 work items
//     in parallel, and lane 0 fills the group's shared-memory stages with 1-D TMA
//     bulk copies (global -> shared, completion counted on the stage's "full"
//     mbarrier);
//   * the consumer warps wait on a stage's full barrier, split the item's rows
//     between them, and release the stage on its "empty" barrier.
// Pipeline g owns the CTA's work items k = g, g + groups, ... and the stages
// g, g + groups, ...; its u-th item uses stage g + groups * (u % stages_per_group).
// A stage is therefore only ever used by one pipeline, in order, so mbarrier
// parity waits are unambiguous. A producer lane needs several hundred cycles to
// issue a tile's copies; with one producer per group the issue rate scales with
// the groups, and an expensive item (a flush) only delays its own pipeline.
//
// Every wait is bounded (RSSM_WAIT_NS, or the policy's Args::wait_ns when it has
// one); a wait that expires sets an abort flag and RSSM_DEVERR_TIMEOUT, and all
// warps wind down: waiting warps give up as soon as the flag is set, and each
// producer, before it exits, waits (bounded again) for the copies it issued into
// stages nobody consumed, so no bulk copy into this CTA's shared memory is left in
// flight when the CTA exits.
//
// A kernel policy K provides:
//   static constexpr int kGroup;          warps per consumer group
//   struct Args  (kernel arguments; must contain int stages, stage_bytes,
//                 stage_off, scratch_off, warp_scratch; int32_t* dev_err)
//   struct Meta  (per-item metadata written by the producer, <= 64 bytes)
//   static __device__ int  n_items(const Args&);
//   static __device__ int4 prefetch(const Args&, int item);     any lane
//   static __device__ void issue(const Args&, int item, int4 info, Meta* meta,
//                                uint8_t* stage, uint64_t* full, uint64_t policy);
//                                (lane 0; arrives on `full` exactly once)
//   static __device__ void consume(const Args&, int item, const Meta&,
//                                  const uint8_t* stage, uint8_t* scratch, int lane,
//                                  int wi);   (whole consumer warp; wi = warp in group)
#pragma once

#include "common.cuh"
#include "internal.h"

namespace rssm {

constexpr int kPipeMaxStages = 16;
constexpr int kPipeMetaBytes = 64;
constexpr int kPipeMaxGroups = 4;
constexpr int kPipeHeader = 2048;  // barriers + metadata + control, before the scratch
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void mbar_arrive_plain(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// The wait limit of a policy: Args::wait_ns when the policy has it, else RSSM_WAIT_NS.
template <class K, class = void>
struct WaitLimit {
    static __device__ __forceinline__ uint64_t ns(const typename K::Args&) { return RSSM_WAIT_NS; }
};
template <class K>
struct WaitLimit<K, decltype(void(K::Args::wait_ns))> {
    static __device__ __forceinline__ uint64_t ns(const typename K::Args& a) { return a.wait_ns; }
};

template <class K>
__global__ void __launch_bounds__(32 * kPipeMaxGroups * (K::kGroup + 1), 1)
    pipe_kernel(const typename K::Args a) {
    extern __shared__ __align__(128) uint8_t smem[];
    static_assert(sizeof(typename K::Meta) <= kPipeMetaBytes, "meta too large");
    uint64_t* fullb = reinterpret_cast<uint64_t*>(smem);
    uint64_t* emptyb = fullb + kPipeMaxStages;
    uint8_t* meta_base = smem + 256;
    volatile int* abort_flag =
        reinterpret_cast<volatile int*>(smem + 256 + kPipeMaxStages * kPipeMetaBytes);
    uint8_t* stage0 = smem + a.stage_off;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ng = (blockDim.x >> 5) / (K::kGroup + 1);  // pipelines
    const int nc = ng * K::kGroup;                        // consumer warps come first
    const int NST = a.stages;
    const int spg = NST / ng;  // stages per pipeline
    const int n = K::n_items(a);
    auto meta_of = [&](int st) {
        return reinterpret_cast<typename K::Meta*>(meta_base + st * kPipeMetaBytes);
    };

    if (threadIdx.x == 0) {
        for (int st = 0; st < NST; ++st) {
            mbar_init(&fullb[st], 1);
            mbar_init(&emptyb[st], K::kGroup);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const uint64_t wait_ns = WaitLimit<K>::ns(a);

    if (warp >= nc) {
        // ---------------- producer warp of pipeline g ----------------
        const int g = warp - nc;
        const uint64_t pol = policy_evict_first();
        int pos = 0, lap = 0;  // stage position and lap of the next item to issue
        for (int u0 = 0;; u0 += 32) {
            const int my_item = blockIdx.x + (g + (u0 + lane) * ng) * gridDim.x;
            int4 info = make_int4(0, 0, 0, 0);
            if (my_item < n) info = K::prefetch(a, my_item);
            int stop = 0;
            for (int j = 0; j < 32; ++j) {
                const int item = blockIdx.x + (g + (u0 + j) * ng) * gridDim.x;
                if (item >= n) {
                    stop = 1;
                    break;
                }
                int4 r;
                r.x = __shfl_sync(kFull, info.x, j);
                r.y = __shfl_sync(kFull, info.y, j);
                r.z = __shfl_sync(kFull, info.z, j);
                r.w = __shfl_sync(kFull, info.w, j);
                int bad = 0;
                if (lane == 0) {
                    const int st = g + ng * pos;
                    int ok = 1;
                    if (lap > 0) ok = mbar_wait_abortable(&emptyb[st], (lap - 1) & 1, wait_ns, abort_flag);
                    if (ok == 0) {
                        *abort_flag = 1;
                        set_dev_err(a.dev_err, RSSM_DEVERR_TIMEOUT);
                    }
                    if (ok != 1 || *abort_flag)
                        bad = 1;
                    else
                        K::issue(a, item, r, meta_of(st), stage0 + (size_t)st * a.stage_bytes,
                                 &fullb[st], pol);
                }
                if (__shfl_sync(kFull, bad, 0)) {
                    stop = 1;
                    break;
                }
                if (++pos == spg) {
                    pos = 0;
                    ++lap;
                }
            }
            if (stop) break;
        }
        // Wind-down after an abort: the last issue into each stage may still have copies
        // in flight if no consumer waited for it. Stage position p has had
        // lap + (p < pos) issues; wait (bounded) for the phase of the last one.
        if (lane == 0 && *abort_flag) {
            for (int p = 0; p < spg; ++p) {
                const int cnt = lap + (p < pos ? 1 : 0);
                if (cnt > 0) mbar_wait_bounded(&fullb[g + ng * p], (cnt - 1) & 1, wait_ns);
            }
        }
        return;
    }

    // ---------------- consumer warps of pipeline g ----------------
    uint8_t* scratch = smem + a.scratch_off + warp * a.warp_scratch;
    const int g = warp / K::kGroup, wi = warp % K::kGroup;
    int pos = 0, lap = 0;
    for (int u = 0;; ++u) {
        const int item = blockIdx.x + (g + u * ng) * gridDim.x;
        if (item >= n) break;
        const int st = g + ng * pos;
        const int ok = mbar_wait_abortable(&fullb[st], lap & 1, wait_ns, abort_flag);
        if (__ballot_sync(kFull, ok == 1) != kFull) {
            // a copy did not land in time (or another warp gave up): stop; the producer
            // drains what it issued
            if (__ballot_sync(kFull, ok == 0) && lane == 0) {
                *abort_flag = 1;
                set_dev_err(a.dev_err, RSSM_DEVERR_TIMEOUT);
            }
            break;
        }
        const typename K::Meta m = *meta_of(st);
        K::consume(a, item, m, stage0 + (size_t)st * a.stage_bytes, scratch, lane, wi);
        __syncwarp();
        if (lane == 0) mbar_arrive_plain(&emptyb[st]);
        if (++pos == spg) {
            pos = 0;
            ++lap;
        }
        if (*abort_flag) break;
    }
}

// Host side: pick the pipeline shape, raise the shared-memory limit once, launch
// one CTA per SM (fewer when there are fewer items).
template <class K>
int launch_pipe(typename K::Args a, int stage_bytes, int warp_scratch, int tile_bytes, long n_items,
                cudaStream_t stream) {
    if (n_items <= 0) return RSSM_OK;
    DeviceInfo di;
    if (!device_info(&di)) return RSSM_ERR_CUDA;
    PipeCfg pc;
    if (!pick_pipe(di, stage_bytes, warp_scratch, tile_bytes, kPipeHeader, kPipeMaxStages,
                   K::kGroup, kPipeMaxGroups, &pc))
        return RSSM_ERR_UNSUPPORTED;
    a.stages = pc.stages;
    a.stage_bytes = stage_bytes;
    a.stage_off = pc.stage_off;
    a.scratch_off = pc.scratch_off;
    a.warp_scratch = warp_scratch;
    const void* kfn = reinterpret_cast<const void*>(pipe_kernel<K>);
    if (!ensure_smem_limit(kfn, pc.smem_bytes)) return RSSM_ERR_CUDA;
    long grid = di.sm_count;
    if (grid > n_items) grid = n_items;
    pipe_kernel<K><<<(int)grid, 32 * pc.groups * (K::kGroup + 1), pc.smem_bytes, stream>>>(a);
    return launch_status();
}

}  // namespace rssm
