// common.cuh -- device helpers shared by the ReplaySSM kernels (sm_103a).
//
// * 1-D TMA bulk copies (cp.async.bulk) global -> shared, completing on an
//   mbarrier transaction count; no cluster multicast anywhere.
// * mbarrier waits bounded by %globaltimer: a wait that does not complete within
//   RSSM_WAIT_NS sets RSSM_DEVERR_TIMEOUT and the kernel winds down instead of
//   spinning forever.
// * bfloat16 <-> float32 packing (bf16 is the top half of a float32; widening is
//   exact, narrowing uses the round-to-nearest-even intrinsic).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "rssm.h"

#define RSSM_WAIT_NS 2000000000ull  // 2 s

namespace rssm {

// ----------------------------------------------------------------------------
// shared-memory addresses, mbarriers, bulk copies
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// One arrival on `bar` (no transaction bytes).
__device__ __forceinline__ void mbar_arrive_plain(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Raise the transaction count the current phase of `bar` waits for, without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar` to complete; false when `limit_ns` elapsed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = RSSM_WAIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// As mbar_wait_bounded, but also gives up as soon as *abort is set by another warp.
// Returns 1 (phase completed), 0 (limit elapsed) or -1 (aborted).
__device__ __forceinline__ int mbar_wait_abortable(uint64_t* bar, uint32_t parity,
                                                   uint64_t limit_ns, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return 1;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return 1;
        if (*abort) return -1;
        if (global_ns() - t0 > limit_ns) return 0;
    }
}

// L2 policy: the checkpoint tiles are read once per step; let them leave L2
// first so rings, tables and per-row inputs stay resident.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
        "%2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 2-D TMA tensor copy global -> shared of one box at element coordinates (x, y) of
// the tensor map `tmap` (a __grid_constant__ kernel parameter), completion counted
// on `bar`. x times the element size is a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 2-D TMA tensor copy shared -> global of one box at (x, y) (x, y >= 0), in this
// thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const void* tmap, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     tmap),
                 "r"(x), "r"(y), "r"(smem_addr(src))
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until this thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory stores visible to the async proxy
// (TMA stores and tensor-core operand reads go through it).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_count(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void set_dev_err(int32_t* dev_err, int bit) {
    if (dev_err) atomicOr(dev_err, bit);
}

// ----------------------------------------------------------------------------
// bfloat16 / float32 element access
// ----------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

__device__ __forceinline__ uint16_t f_to_bf16(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return uint32_t(f_to_bf16(lo)) | (uint32_t(f_to_bf16(hi)) << 16);
}

// Load 8 consecutive elements (bf16 when is_bf16, else f32) starting at p (16-byte
// aligned for bf16, 32-byte for f32) into f[0..7].
__device__ __forceinline__ void load8(const void* p, bool is_bf16, float* f) {
    if (is_bf16) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
        const float4 a = reinterpret_cast<const float4*>(p)[0];
        const float4 b = reinterpret_cast<const float4*>(p)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
}

__device__ __forceinline__ void store8(void* p, bool is_bf16, const float* f) {
    if (is_bf16) {
        uint4 v;
        v.x = pack_bf16x2(f[0], f[1]); v.y = pack_bf16x2(f[2], f[3]);
        v.z = pack_bf16x2(f[4], f[5]); v.w = pack_bf16x2(f[6], f[7]);
        *reinterpret_cast<uint4*>(p) = v;
    } else {
        reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
}

// acc + sum_{j<8} s_j c_j for 8 bf16 pairs packed in two uint4: each product is
// formed from the bf16 operands by a mixed-precision fma (f32 accumulate, one
// rounding per step), so no widening instruction is needed.
__device__ __forceinline__ float dot8_bf16(const uint4 s, const uint4 c, float acc) {
    asm("{\n\t.reg .b16 a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3, b4, b5, b6, b7;\n\t"
        "mov.b32 {a0, a1}, %1;\n\tmov.b32 {a2, a3}, %2;\n\t"
        "mov.b32 {a4, a5}, %3;\n\tmov.b32 {a6, a7}, %4;\n\t"
        "mov.b32 {b0, b1}, %5;\n\tmov.b32 {b2, b3}, %6;\n\t"
        "mov.b32 {b4, b5}, %7;\n\tmov.b32 {b6, b7}, %8;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %0, a1, b1, %0;\n\t"
        "fma.rn.f32.bf16 %0, a2, b2, %0;\n\tfma.rn.f32.bf16 %0, a3, b3, %0;\n\t"
        "fma.rn.f32.bf16 %0, a4, b4, %0;\n\tfma.rn.f32.bf16 %0, a5, b5, %0;\n\t"
        "fma.rn.f32.bf16 %0, a6, b6, %0;\n\tfma.rn.f32.bf16 %0, a7, b7, %0;\n\t}"
        : "+f"(acc)
        : "r"(s.x), "r"(s.y), "r"(s.z), "r"(s.w), "r"(c.x), "r"(c.y), "r"(c.z), "r"(c.w));
    return acc;
}

// 16-byte asynchronous copy global -> shared without registers (cp.async, L2 only),
// its group commit and the wait for all of this thread's copies.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float load1(const void* base, long idx, bool is_bf16) {
    return is_bf16 ? bf16_to_f(reinterpret_cast<const uint16_t*>(base)[idx])
                   : reinterpret_cast<const float*>(base)[idx];
}

// 4 consecutive elements (bf16 when bf, else f32) at element index i of base
// (8-byte aligned for bf16, 16-byte for f32) into f[0..3].
__device__ __forceinline__ void load4(const void* base, int i, bool bf, float* f) {
    if (bf) {
        const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + i);
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    } else {
        const float4 v = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
}

__device__ __forceinline__ void store1(void* base, long idx, bool is_bf16, float v) {
    if (is_bf16) reinterpret_cast<uint16_t*>(base)[idx] = f_to_bf16(v);
    else reinterpret_cast<float*>(base)[idx] = v;
}

// ----------------------------------------------------------------------------
// counter-based random bits and stochastic rounding to bfloat16
// ----------------------------------------------------------------------------

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC 2011): ten rounds of two 32x32->64 multiplies whose high halves are
// xor-ed with the other counter words and the key, the key bumped by the Weyl
// increments between rounds. Returns four 32-bit words for counter c, key k.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        // one widening multiply gives both halves of each product
        const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c.x;
        const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
        c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ k.x, static_cast<uint32_t>(p1),
                       static_cast<uint32_t>(p0 >> 32) ^ c.w ^ k.y, static_cast<uint32_t>(p0));
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// Stochastic rounding of a float32 to bfloat16 with 16 random bits r: adding r to
// the 16 bits that bfloat16 drops and truncating rounds away from zero with
// probability (dropped bits) / 2^16, so the rounding is unbiased. Inf and NaN keep
// round-to-nearest.
__device__ __forceinline__ uint16_t f_to_bf16_sr(float f, uint32_t r) {
    const uint32_t u = __float_as_uint(f);
    if ((u & 0x7f800000u) == 0x7f800000u) return f_to_bf16(f);
    return static_cast<uint16_t>((u + (r & 0xFFFFu)) >> 16);
}

// 8 float32 values as bfloat16 with stochastic rounding; the random bits are
// Philox4x32-10 at counter (group, offset), key seed, where group numbers the
// 8-element groups of the destination array.
__device__ __forceinline__ uint4 pack8_bf16_sr(const float* f, uint64_t group, uint64_t seed,
                                               uint64_t offset) {
    const uint4 r = philox4x32_10(
        make_uint4((uint32_t)group, (uint32_t)(group >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)),
        make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint4 v;
    uint32_t* o = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = uint32_t(f_to_bf16_sr(f[2 * i], w[i])) | (uint32_t(f_to_bf16_sr(f[2 * i + 1], w[i] >> 16)) << 16);
    return v;
}

// Store 8 float32 values as bfloat16 at p (16-byte aligned) with stochastic rounding
// (bits as pack8_bf16_sr).
__device__ __forceinline__ void store8_bf16_sr(void* p, const float* f, uint64_t group,
                                               uint64_t seed, uint64_t offset) {
    *reinterpret_cast<uint4*>(p) = pack8_bf16_sr(f, group, seed, offset);
}

// State element types for templated kernels (sr: stores round stochastically).
struct StF32 {
    static constexpr int bytes = 4;
    static constexpr bool bf16 = false;
    static constexpr bool sr = false;
};
struct StBF16 {
    static constexpr int bytes = 2;
    static constexpr bool bf16 = true;
    static constexpr bool sr = false;
};
struct StBF16SR {
    static constexpr int bytes = 2;
    static constexpr bool bf16 = true;
    static constexpr bool sr = true;
};

// softplus(x) = log(1 + e^x); above 20 the correction is below float32 resolution.
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }
// The same gate through the fast exponential and division intrinsics (a few ulp):
// for per-draft epilogues where the accurate path's latency shows.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// ----------------------------------------------------------------------------
// warp reduce-scatter
// ----------------------------------------------------------------------------

// `v[0..CNT)` holds partial sums on each lane of a group of GRP consecutive lanes
// (GRP a power of two <= 32, CNT a power of two <= GRP). Afterwards v[0] on every
// lane holds the group total of entry index `out_idx` (returned), where lanes
// whose low bits (below GRP/CNT) differ hold the same entry.
template <int CNT, int GRP>
__device__ __forceinline__ int reduce_scatter(float* v) {
    static_assert((CNT & (CNT - 1)) == 0 && (GRP & (GRP - 1)) == 0 && CNT <= GRP, "shape");
    const int lane = threadIdx.x & 31;
    int idx = 0;
    int c = CNT;
#pragma unroll
    for (int o = GRP / 2; o >= 1; o >>= 1) {
        if (c > 1) {
            const bool upper = (lane & o) != 0;
            const int h = c / 2;
#pragma unroll
            for (int i = 0; i < CNT / 2; ++i) {
                if (i < h) {
                    const float send = upper ? v[i] : v[i + h];
                    const float keep = upper ? v[i + h] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            if (upper) idx += h;
            c = h;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
    return idx;
}

}  // namespace rssm
