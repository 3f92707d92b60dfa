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
#include "umma.cuh"

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

// The tensor-core fold on its own: D[r][c] = sum_{i<=w} A[r][i] B[i][c] for 128 rows,
// with A float32 (split into three bf16 parts, K = 48 in three MMAs of K = 16) and B
// the bf16 ring layout [16][N] (entries above w ignored), D read back from TMEM by
// the four warps (warp q owns rows 32q..32q+31). One CTA of 128 threads.
constexpr int kFoldK = 16;
constexpr uint32_t kALbo = 128, kASbo = 6 * 128;   // A: 128 rows x 48 (3 splits x 16)
constexpr uint32_t kBLbo = 128, kBSbo = 2 * 128;   // B^T: N rows x 16

template <int N>
__global__ void __launch_bounds__(128, 1)
    umma_fold_kernel(const float* A, const uint16_t* B, int w, float* D, int32_t* dev_err) {
    __shared__ __align__(1024) uint8_t sA[16 * kASbo];
    __shared__ __align__(1024) uint8_t sB[(N / 8) * kBSbo];
    __shared__ __align__(16) uint16_t sRing[kFoldK * N];
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    if (warp == 0) umma::tmem_alloc(&tbase, N < 32 ? 32 : N);
    if (t == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    // ring entries 0..w, zeros above
    for (int e = t; e < kFoldK * N; e += 128) sRing[e] = (e / N <= w) ? B[e] : (uint16_t)0;
    // A: row t, entries 0..15 (zero above w), three bf16 parts side by side along K
    {
        uint16_t part[3][kFoldK];
#pragma unroll
        for (int i = 0; i < kFoldK; ++i) {
            const float x = i <= w ? A[t * kFoldK + i] : 0.f;
            umma::split3_bf16(x, part[0][i], part[1][i], part[2][i]);
        }
#pragma unroll
        for (int sp = 0; sp < 3; ++sp)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 v;
                v.x = part[sp][8 * h] | (uint32_t(part[sp][8 * h + 1]) << 16);
                v.y = part[sp][8 * h + 2] | (uint32_t(part[sp][8 * h + 3]) << 16);
                v.z = part[sp][8 * h + 4] | (uint32_t(part[sp][8 * h + 5]) << 16);
                v.w = part[sp][8 * h + 6] | (uint32_t(part[sp][8 * h + 7]) << 16);
                *reinterpret_cast<uint4*>(sA + umma::kmajor_offset(t, 16 * sp + 8 * h, kALbo, kASbo)) = v;
            }
    }
    __syncthreads();
    // B^T: block (n-block nb, k-block kb) = transpose of ring rows 8kb.. x columns 8nb..
    if (t < (N / 8) * 2) {
        const int nb = t % (N / 8), kb = t / (N / 8);
        uint4 in[8], out[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
            in[r] = *reinterpret_cast<const uint4*>(sRing + (8 * kb + r) * N + 8 * nb);
        umma::transpose8x8_b16(in, out);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sB + umma::kmajor_offset(8 * nb + c, 8 * kb, kBLbo, kBSbo)) = out[c];
    }
    umma::fence_smem_to_async();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t d_tmem = tbase;
    if (t == 0) {
        const uint32_t idesc = umma::idesc_bf16_f32(128, N);
        const uint64_t bdesc = umma::smem_desc_kmajor(sB, kBLbo, kBSbo);
#pragma unroll
        for (int sp = 0; sp < 3; ++sp)
            umma::mma_bf16(d_tmem, umma::smem_desc_kmajor(sA + sp * 2 * kALbo, kALbo, kASbo), bdesc,
                           idesc, sp > 0);
        umma::commit_to(&bar);
    }
    const bool ok = mbar_wait_bounded(&bar, 0);
    if (!ok && lane == 0) set_dev_err(dev_err, RSSM_DEVERR_TIMEOUT);
    umma::fence_after_sync();
    if (ok) {
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            umma::ld32(d_tmem + ((uint32_t)(32 * warp) << 16) + c0, v);
            umma::wait_ld();
            const int row = 32 * warp + lane;
#pragma unroll
            for (int j = 0; j < 32; ++j) D[row * N + c0 + j] = v[j];
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(d_tmem, N < 32 ? 32 : N);
}

}  // namespace dbg
}  // namespace rssm

using namespace rssm;

extern "C" int rssm_debug_umma_fold(const float* A, const uint16_t* B, int w, int N, float* D,
                                    int32_t* dev_err, rssm_stream_t stream) {
    if (w < 0 || w >= dbg::kFoldK || (N != 64 && N != 128)) return RSSM_ERR_INVALID_ARG;
    if (!ok_ptr(A) || !ok_ptr(B) || !ok_ptr(D)) return RSSM_ERR_INVALID_ARG;
    if (N == 128)
        dbg::umma_fold_kernel<128><<<1, 128, 0, (cudaStream_t)stream>>>(A, B, w, D, dev_err);
    else
        dbg::umma_fold_kernel<64><<<1, 128, 0, (cudaStream_t)stream>>>(A, B, w, D, dev_err);
    return launch_status();
}

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
