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
#include "umma.cuh"

namespace rssm {

constexpr int kPipeMaxStages = 16;
constexpr int kPipeMetaBytes = 64;
constexpr int kPipeMaxGroups = 4;
constexpr int kPipeHeader = 2048;  // barriers + metadata + control, before the scratch
constexpr unsigned kFull = 0xffffffffu;


// Tensor memory: a policy with `static constexpr int kTmemCols > 0` gets that many
// TMEM columns (allocated by consumer warp 0 when the CTA starts, freed when every
// consumer warp is done). A policy with kTmemCols > 0 or `kUsesCtx = true` gets a
// PipeCtx as the last argument of consume(): per consumer group a tensor-core
// completion mbarrier, a hand-over mbarrier (one arrival per warp) and a "taken"
// mbarrier (one arrival), and the means to release the stage itself.
template <class K, class = void>
struct TmemCols {
    static constexpr int value = 0;
};
template <class K>
struct TmemCols<K, decltype(void(K::kTmemCols))> {
    static constexpr int value = K::kTmemCols;
};

// Dynamic work distribution: a policy with `static constexpr bool kDynamic = true` and
// an Args member `unsigned int* sched` (two words, zero before the launch) has its
// producers claim kClaim items at a time from the counter sched[0] instead of taking
// every (gridDim.x * groups)-th item, so consumer groups that met expensive items take
// fewer. Each producer ends its pipeline with an end marker (item -1) and then counts
// itself in sched[1]; the last producer of the launch sets both words back to zero.
template <class K, class = void>
struct DynSched {
    static constexpr bool value = false;
};
template <class K>
struct DynSched<K, decltype(void(K::kDynamic))> {
    static constexpr bool value = K::kDynamic;
};
constexpr int kClaim = 2;

template <class K, class = void>
struct UsesCtx {
    static constexpr bool value = TmemCols<K>::value > 0;
};
template <class K>
struct UsesCtx<K, decltype(void(K::kUsesCtx))> {
    static constexpr bool value = K::kUsesCtx || TmemCols<K>::value > 0;
};

struct PipeCtx {
    uint32_t tmem;       // TMEM base address of the CTA's allocation
    uint64_t* mma_bar;   // this group's tensor-core completion barrier (one commit)
    uint64_t* grp_bar;   // this group's hand-over barrier (one arrival per warp)
    uint64_t* done_bar;  // the issuing thread has taken a hand-over (one arrival)
    uint32_t mma_phase;  // parities of those barriers' next completions (the policy
    uint32_t grp_phase;  // flips them as it uses them)
    uint32_t done_phase;
    int group;           // consumer group index
    int groups;          // consumer groups in the CTA
    volatile int* abort_flag;
    uint64_t* empty_bar;  // the current stage's "empty" barrier
    bool released;        // the policy already gave the stage back (release_stage)
};

// Give the current stage back to the producer before consume() returns: the policy
// must not touch the stage's shared memory afterwards. Whole warp.
__device__ __forceinline__ void release_stage(PipeCtx& ctx) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(
                                                  smem_addr(ctx.empty_bar))
                                              : "memory");
    ctx.released = true;
}

constexpr int kPipeTmemSlot = 1296;  // header offsets: TMEM base address,
constexpr int kPipeMmaBars = 1312;   // the groups' completion barriers,
constexpr int kPipeGrpBars = 1344;   // their hand-over barriers,
constexpr int kPipeDoneBars = 1376;  // their "taken" barriers,
constexpr int kPipeItems = 1408;     // and (dynamic distribution) each stage's item

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
    pipe_kernel(const __grid_constant__ typename K::Args a) {
    extern __shared__ __align__(1024) uint8_t smem[];
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

    constexpr int kTmem = TmemCols<K>::value;
    constexpr bool kCtx = UsesCtx<K>::value;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kPipeTmemSlot);
    uint64_t* mma_bars = reinterpret_cast<uint64_t*>(smem + kPipeMmaBars);
    uint64_t* grp_bars = reinterpret_cast<uint64_t*>(smem + kPipeGrpBars);
    uint64_t* done_bars = reinterpret_cast<uint64_t*>(smem + kPipeDoneBars);
    if constexpr (kTmem > 0) {
        if (warp == 0) umma::tmem_alloc(tmem_slot, kTmem);
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < NST; ++st) {
            mbar_init(&fullb[st], 1);
            mbar_init(&emptyb[st], K::kGroup);
        }
        if constexpr (kCtx)
            for (int g = 0; g < ng; ++g) {
                mbar_init(&mma_bars[g], 1);
                mbar_init(&grp_bars[g], K::kGroup);
                mbar_init(&done_bars[g], 1);
            }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if constexpr (kTmem > 0) umma::fence_before_sync();
    __syncthreads();

    const uint64_t wait_ns = WaitLimit<K>::ns(a);

    constexpr bool kDyn = DynSched<K>::value;
    volatile int* stage_item = reinterpret_cast<volatile int*>(smem + kPipeItems);

    if (warp >= nc) {
        // ---------------- producer warp of pipeline g ----------------
        const int g = warp - nc;
        const uint64_t pol = policy_evict_first();
        int pos = 0, lap = 0;  // stage position and lap of the next item to issue
        if constexpr (kDyn) {
            // About three quarters of the items are dealt round-robin as in the static
            // scheme (producer (block, g) takes items block + (g + u * groups) * gridDim.x
            // for u < U, in order, with no atomic before its first copy); the rest are
            // claimed kClaim at a time from the counter, the next claim made while the
            // current one issues. The counter thus only balances the tail of the launch,
            // where differences between groups add up, with few atomics.
            const int stride = (int)(gridDim.x * ng);
            const int U = (3 * n / 4) / stride;
            const int first = U * stride;
            int u = 0;
            int base = U > 0 ? (int)blockIdx.x + g * (int)gridDim.x : 0;
            if (U == 0) {
                if (lane == 0) base = first + (int)atomicAdd(a.sched, (unsigned)kClaim);
                base = __shfl_sync(kFull, base, 0);
            }
            for (bool stop = false; !stop;) {
                // this round: one static item (u < U) or kClaim claimed ones
                const bool stat = u < U;
                const int cnt = stat ? 1 : kClaim;
                int nxt = 0;
                if (u + 1 < U) nxt = (int)blockIdx.x + (g + (u + 1) * ng) * (int)gridDim.x;
                else if (lane == 0 && base < n) nxt = first + (int)atomicAdd(a.sched, (unsigned)kClaim);
                ++u;
                int4 info = make_int4(0, 0, 0, 0);
                if (lane < cnt && base + lane < n) info = K::prefetch(a, base + lane);
                for (int j = 0; j < cnt && !stop; ++j) {
                    const int item = base + j;
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
                        if (ok != 1 || *abort_flag) {
                            bad = 1;
                        } else if (item >= n) {
                            stage_item[st] = -1;  // end marker
                            mbar_arrive_plain(&fullb[st]);
                        } else {
                            stage_item[st] = item;
                            K::issue(a, item, r, meta_of(st), stage0 + (size_t)st * a.stage_bytes,
                                     &fullb[st], pol);
                        }
                    }
                    if (__shfl_sync(kFull, bad, 0)) {
                        stop = true;
                        break;
                    }
                    if (++pos == spg) {
                        pos = 0;
                        ++lap;
                    }
                    if (item >= n) stop = true;
                }
                base = __shfl_sync(kFull, nxt, 0);
            }
        } else {
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
        if constexpr (kDyn) {
            // every producer has made its last claim once all have counted themselves:
            // the last one resets the counter for the next launch
            if (lane == 0) {
                __threadfence();
                const unsigned prev = atomicAdd(a.sched + 1, 1u);
                if (prev == gridDim.x * (unsigned)ng - 1u) {
                    atomicExch(a.sched, 0u);
                    atomicExch(a.sched + 1, 0u);
                    __threadfence();
                }
            }
        }
        return;
    }

    // ---------------- consumer warps of pipeline g ----------------
    uint8_t* scratch = smem + a.scratch_off + warp * a.warp_scratch;
    const int g = warp / K::kGroup, wi = warp % K::kGroup;
    PipeCtx ctx{};
    if constexpr (kCtx) {
        if constexpr (kTmem > 0) {
            umma::fence_after_sync();
            ctx.tmem = *tmem_slot;
        }
        ctx.mma_bar = &mma_bars[g];
        ctx.grp_bar = &grp_bars[g];
        ctx.done_bar = &done_bars[g];
        ctx.mma_phase = 0;
        ctx.grp_phase = 0;
        ctx.done_phase = 0;
        ctx.group = g;
        ctx.groups = ng;
        ctx.abort_flag = abort_flag;
    }
    int pos = 0, lap = 0;
    for (int u = 0;; ++u) {
        int item = blockIdx.x + (g + u * ng) * gridDim.x;
        if (!kDyn && item >= n) break;
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
        if constexpr (kDyn) {
            item = stage_item[st];
            if (item < 0) break;  // end marker: no more items for this pipeline
        }
        const typename K::Meta m = *meta_of(st);
        if constexpr (kCtx) {
            ctx.empty_bar = &emptyb[st];
            ctx.released = false;
            K::consume(a, item, m, stage0 + (size_t)st * a.stage_bytes, scratch, lane, wi, ctx);
        } else {
            K::consume(a, item, m, stage0 + (size_t)st * a.stage_bytes, scratch, lane, wi);
        }
        __syncwarp();
        if constexpr (kCtx) {
            if (!ctx.released && lane == 0) mbar_arrive_plain(&emptyb[st]);
        } else {
            if (lane == 0) mbar_arrive_plain(&emptyb[st]);
        }
        if (++pos == spg) {
            pos = 0;
            ++lap;
        }
        if (*abort_flag) break;
    }
    if constexpr (kTmem > 0) {
        // every consumer warp is done with tensor memory: warp 0 frees it
        umma::fence_before_sync();
        umma::named_sync(15, nc * 32);
        if (warp == 0) {
            umma::fence_after_sync();
            umma::tmem_dealloc(ctx.tmem, kTmem);
        }
    }
}

// Host side: pick the pipeline shape, raise the shared-memory limit once, launch
// one CTA per SM (fewer when there are fewer items).
// `align`: alignment of the stages' start (1024 for 128-byte-swizzled TMA boxes; the
// stage size is then a multiple of it too).
template <class K>
int launch_pipe(typename K::Args a, int stage_bytes, int warp_scratch, int tile_bytes, long n_items,
                cudaStream_t stream, int align = 128) {
    if (n_items <= 0) return RSSM_OK;
    DeviceInfo di;
    if (!device_info(&di)) return RSSM_ERR_CUDA;
    PipeCfg pc;
    if (!pick_pipe(di, stage_bytes, warp_scratch, tile_bytes, kPipeHeader, kPipeMaxStages,
                   K::kGroup, kPipeMaxGroups, &pc, align))
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
