// umma.cuh -- 5th-generation tensor-core (tcgen05) building blocks for sm_103a.
//
// Used by the flush folds: a fold of w + 1 ring entries into a checkpoint tile is
// the dense product D[r][c] = sum_i A[r][i] B[i][c] (rows r of the tile, columns c,
// ring entries i), which one tcgen05.mma per K = 16 entries computes into a tensor-
// memory (TMEM) accumulator. What is here:
//   * TMEM allocation (tcgen05.alloc / dealloc, one warp) and the fences that order
//     tcgen05 operations around thread synchronisation;
//   * shared-memory matrix descriptors for the K-major layout without swizzling:
//     the operand is made of "core matrices" of 8 rows x 16 bytes (8 bf16 along K),
//     each stored as 128 contiguous bytes; LBO is the byte distance between core
//     matrices adjacent along K, SBO between core matrices adjacent along M (or N);
//   * the instruction descriptor of kind::f16 (bf16 x bf16 -> f32, both K-major);
//   * the MMA itself (issued by one thread), its commit to an mbarrier, and the
//     32x32b TMEM load (warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace rssm {
namespace umma {

// ---------------------------------------------------------------- TMEM ----

// Allocate `ncols` TMEM columns (a power of two >= 32) for this CTA; the base
// address is written to *smem_dst. Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(smem_dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Free what tmem_alloc took. Whole warp (the one that allocated).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory stores visible to the async proxy
// (the tensor core reads operands through it).
__device__ __forceinline__ void fence_smem_to_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------- descriptors ----

// K-major operand, no swizzle: core matrix (m-block mb, k-block kb) at
// start + mb * sbo + kb * lbo, 128 contiguous bytes (8 rows of 16 bytes).
__device__ __forceinline__ uint64_t smem_desc_kmajor(const void* start, uint32_t lbo, uint32_t sbo) {
    const uint64_t a = smem_addr(start);
    uint64_t d = 0;
    d |= (a >> 4) & 0x3FFFull;                       // bits 0-13: start address / 16
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;      // bits 16-29: leading byte offset / 16
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;      // bits 32-45: stride byte offset / 16
    d |= 1ull << 46;                                 // bits 46-47: descriptor version 1
    // base offset 0, relative LBO, layout type 0 (no swizzle)
    return d;
}

// Byte offset of element (r, k) (bf16) inside a K-major no-swizzle operand.
__host__ __device__ __forceinline__ uint32_t kmajor_offset(int r, int k, uint32_t lbo, uint32_t sbo) {
    return (uint32_t)(r >> 3) * sbo + (uint32_t)(k >> 3) * lbo + (uint32_t)(r & 7) * 16u +
           (uint32_t)(k & 7) * 2u;
}

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, no negation,
// dense, shape M x N (M in {64, 128}, N a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                          // D format: f32
           | (1u << 7)                        // A format: bf16
           | (1u << 10)                       // B format: bf16
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// ------------------------------------------------------------------ MMA ----

// D[tmem] (+)= A[smem] * B[smem]^T-as-described, one K = 16 step. One thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far completes.
__device__ __forceinline__ void commit_to(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

// -------------------------------------------------------------- TMEM load ----

// 32 consecutive 32-bit columns of this thread's TMEM lane (warp-collective; the
// lane is 32 (warp % 4) + laneid, `taddr` carries the warp's lane base in bits
// 16-31). Call wait_ld() before using the values.
__device__ __forceinline__ void ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive 32-bit columns of this thread's TMEM lane (two 32x32b.x32 loads
// issued back to back; one wait covers both).
__device__ __forceinline__ void ld64(uint32_t taddr, float* v) {
    ld32(taddr, v);
    ld32(taddr + 32, v + 32);
}

__device__ __forceinline__ void wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Store 32 consecutive 32-bit columns of this thread's TMEM lane (warp-collective,
// lane addressing as ld32). Call wait_st() before anything that depends on it.
__device__ __forceinline__ void st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------- bf16 splitting ----

// x = hi + mid + lo with each part a bf16 (x's float32 significand, 24 bits, is
// carried by three 8-bit parts; the remainders are exact in float32).
__device__ __forceinline__ void split3_bf16(float x, uint16_t& hi, uint16_t& mid, uint16_t& lo) {
    hi = f_to_bf16(x);
    const float r1 = x - bf16_to_f(hi);
    mid = f_to_bf16(r1);
    lo = f_to_bf16(r1 - bf16_to_f(mid));
}

// Transpose an 8 x 8 block of 16-bit values held as 8 rows of 8 (uint4 each) into
// its columns.
__device__ __forceinline__ void transpose8x8_b16(const uint4 (&in)[8], uint4 (&out)[8]) {
    // element (r, c) is half (c & 1) of word (c >> 1) of in[r]
    uint32_t w[8][4];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        w[r][0] = in[r].x; w[r][1] = in[r].y; w[r][2] = in[r].z; w[r][3] = in[r].w;
    }
    uint32_t o[8][4];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        // out row c = (in[0][c], in[1][c], ..., in[7][c])
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a = w[2 * j][c >> 1], b = w[2 * j + 1][c >> 1];
            // low half of the result word = element of row 2j, high half = row 2j+1
            o[c][j] = (c & 1) ? __byte_perm(a, b, 0x7632) : __byte_perm(a, b, 0x5410);
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) out[c] = make_uint4(o[c][0], o[c][1], o[c][2], o[c][3]);
}

}  // namespace umma
}  // namespace rssm
