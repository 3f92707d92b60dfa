// mamba2_prologue.cu -- the per-row prologue of a Mamba2 ReplaySSM decode step
// on sm_103a: ring append, coefficient tables, and both fused with the cursor
// step in one launch.
//
// Pages followed: [M2] "ReplaySSM: cache SSM inputs for faster Mamba2 standard
// decode" (vLLM PR 48018 report): 实现拆解 item 1 (a precompute kernel for the
// per-row decay products and B . C scalars), 实现拆解 item 2 (x_cache,
// dt_cache, B_cache written at write_pos), 实现拆解 item 3 (per-row write_pos and
// is_flush computed on the device).
//
// Kernels (one CTA per row):
//   ring_append_kernel  x, dt = softplus(dt_raw + dt_bias), B into ring entry w.
//   precompute_kernel   stages C_t and the slot's whole dt and B rings in shared
//                       memory, then B_i . C_t per group and the decay suffix
//                       products per head, written as per-(row, head) tables.
//   prepare_kernel      cursor step + ring append + tables: the slot's rings are
//                       staged while the cursor is read, entry w is patched from
//                       the step's inputs.
// The tables are latency-bound work on a few tens of KB per row, so every load a
// thread makes is issued before any of its results is used.
#include "common.cuh"
#include "cursor.cuh"
#include "internal.h"
#include "mamba2.cuh"

namespace rssm {
namespace m2 {

// ----------------------------------------------------------------------------
// per-row prologue pieces
// ----------------------------------------------------------------------------

struct RowArgs {
    int H, P, N, G, L, num_slots, act_bf16;
    const void* x;         // [batch][H][P]
    const float* dt_raw;   // [batch][H]
    const float* dt_bias;  // [H] or null
    int softplus;
    const void* B;         // [batch][G][N]
    const float* A;        // [H]
    const void* C;         // [batch][G][N]
    void* ring_x;          // [slots][H][L][P]
    float* ring_dt;        // [slots][H][L]
    void* ring_B;          // [slots][G][L][N]
    float* ws;             // [batch][H][TBL]
};

constexpr int kRowThreads = 512;

// n elements from src to dst; each thread issues four loads before its four stores.
template <class V>
__device__ __forceinline__ void copy4(V* dst, const V* src, int n) {
    for (int base = threadIdx.x; base < n; base += 4 * blockDim.x) {
        V r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = base + u * blockDim.x;
            if (i < n) r[u] = __ldcg(src + i);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = base + u * blockDim.x;
            if (i < n) dst[i] = r[u];
        }
    }
}

__device__ __forceinline__ float step_dt(const RowArgs& a, int b, int h) {
    float v = a.dt_raw[(size_t)b * a.H + h] + (a.dt_bias ? a.dt_bias[h] : 0.f);
    return a.softplus ? softplus_f(v) : v;
}

// Entry w of slot s's rings <- row b's x, dt = softplus(dt_raw + dt_bias), B.
__device__ void append_row(const RowArgs& a, int b, int s, int w) {
    const int H = a.H, P = a.P, N = a.N, G = a.G, L = a.L;
    const int sa = a.act_bf16 ? 2 : 4;
    const int xc = P * sa / 16;  // 16-byte chunks per head row
    const uint4* xs =
        reinterpret_cast<const uint4*>(static_cast<const char*>(a.x) + (size_t)b * H * P * sa);
    for (int c = threadIdx.x; c < H * xc; c += blockDim.x) {
        const int h = c / xc, j = c % xc;
        reinterpret_cast<uint4*>(static_cast<char*>(a.ring_x) + (((size_t)s * H + h) * L + w) * P * sa)[j] =
            xs[c];
    }
    for (int h = threadIdx.x; h < H; h += blockDim.x) a.ring_dt[((size_t)s * H + h) * L + w] = step_dt(a, b, h);
    const int bc = N * sa / 16;
    const uint4* bs =
        reinterpret_cast<const uint4*>(static_cast<const char*>(a.B) + (size_t)b * G * N * sa);
    for (int c = threadIdx.x; c < G * bc; c += blockDim.x) {
        const int g = c / bc, j = c % bc;
        reinterpret_cast<uint4*>(static_cast<char*>(a.ring_B) + (((size_t)s * G + g) * L + w) * N * sa)[j] =
            bs[c];
    }
}

// Shared memory of the table-building kernels, in bytes: C_t [G][N] f32, the dt
// ring [H][L+1] f32 (rows padded to an odd stride), B . C [G][L] f32, the B ring
// [G][L][N] (activation type).
__host__ __device__ inline int prologue_smem(int H, int N, int G, int L, int sa) {
    return ((G * N + H * (L + 1) + G * L + 3) & ~3) * 4 + G * L * N * sa;
}

// Row b's C_t and slot s's whole dt and B rings into shared memory.
__device__ void stage_slot(const RowArgs& a, int b, int s, float* sm) {
    const int H = a.H, N = a.N, G = a.G, L = a.L;
    const bool bf = a.act_bf16;
    const int sa = bf ? 2 : 4;
    float* cs = sm;
    float* dts = cs + G * N;
    char* braw = reinterpret_cast<char*>(sm + ((G * N + H * (L + 1) + G * L + 3) & ~3));
    for (int e = threadIdx.x * 8; e < G * N; e += blockDim.x * 8)
        load8(static_cast<const char*>(a.C) + ((size_t)b * G * N + e) * sa, bf, cs + e);
    const float* dr = a.ring_dt + (size_t)s * H * L;
    for (int base = threadIdx.x; base < H * L; base += 4 * blockDim.x) {
        float r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = base + u * blockDim.x;
            if (i < H * L) r[u] = __ldcg(dr + i);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = base + u * blockDim.x;
            if (i < H * L) dts[(i / L) * (L + 1) + (i - (i / L) * L)] = r[u];
        }
    }
    copy4(reinterpret_cast<uint4*>(braw),
          reinterpret_cast<const uint4*>(static_cast<const char*>(a.ring_B) + (size_t)s * G * L * N * sa),
          G * L * N * sa / 16);
}

// Row b's tables from the staged rings (entries 0..w):
//   P_i = exp(A_h sum_{j>i} dt_j), coef_i = P_i dt_i (B_i . C_t), a_i = P_i dt_i,
//   Pm1 = exp(A_h sum_{j<=w} dt_j), written straight to the workspace.
__device__ void tables_from_smem(const RowArgs& a, int b, int w, float* sm) {
    const int H = a.H, N = a.N, G = a.G, L = a.L;
    const int TBL = tbl_floats(L);
    const bool bf = a.act_bf16;
    const int sa = bf ? 2 : 4;
    const int hpg = H / G;
    const float* cs = sm;
    const float* dts = cs + G * N;
    float* bc = sm + G * N + H * (L + 1);
    const char* braw = reinterpret_cast<const char*>(sm + ((G * N + H * (L + 1) + G * L + 3) & ~3));

    // bc[g][i] = B_i . C_t: one warp per (group, entry), lanes over dstate
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int pair = warp; pair < G * (w + 1); pair += nwarps) {
        const int g = pair / (w + 1), i = pair - (pair / (w + 1)) * (w + 1);
        const char* Bi = braw + ((size_t)g * L + i) * N * sa;
        const float* cg = cs + g * N;
        float acc = 0.f;
        for (int n = lane; n < N; n += 32) acc = fmaf(load1(Bi, n, bf), cg[n], acc);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) bc[g * L + i] = acc;
    }
    __syncthreads();

    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const int g = h / hpg;
        const float* dh = dts + h * (L + 1);
        float* t = a.ws + ((size_t)b * H + h) * TBL;
        const float Ah = a.A[h];
        float suffix = 0.f;
        for (int i = w; i >= 0; --i) {
            const float dti = dh[i];
            const float Pi = expf(Ah * suffix);
            t[i] = Pi * dti * bc[g * L + i];
            t[L + i] = Pi * dti;
            suffix += dti;
        }
        for (int i = w + 1; i < L; ++i) {
            t[i] = 0.f;
            t[L + i] = 0.f;
        }
        t[2 * L] = expf(Ah * suffix);
        for (int i = 2 * L + 1; i < TBL; ++i) t[i] = 0.f;
    }
}

// ----------------------------------------------------------------------------
// prologue kernels
// ----------------------------------------------------------------------------

__global__ void __launch_bounds__(256) ring_append_kernel(const RowArgs a, const int32_t* ci,
                                                          const int32_t* row_wp, int32_t* dev_err) {
    const int b = blockIdx.x;
    const int w = given_cursor(b, ci[b], a.num_slots, a.L, row_wp, threadIdx.x == 0 ? dev_err : nullptr);
    if (w < 0) return;
    append_row(a, b, ci[b], w);
}

__global__ void __launch_bounds__(kRowThreads) precompute_kernel(const RowArgs a, const int32_t* ci,
                                                                 const int32_t* row_wp) {
    extern __shared__ __align__(16) float psm[];
    const int b = blockIdx.x;
    // bad slots and cursors are reported by the append and output kernels
    const int w = given_cursor(b, ci[b], a.num_slots, a.L, row_wp, nullptr);
    if (w < 0) return;
    stage_slot(a, b, ci[b], psm);
    __syncthreads();
    tables_from_smem(a, b, w, psm);
}

// Cursor advance (when `advance`), ring append and tables of one row in one CTA.
// The slot's rings are staged while thread 0 reads the cursor; after the append,
// entry w of the staged copy is patched with the step's dt and B.
__global__ void __launch_bounds__(kRowThreads) prepare_kernel(const RowArgs a, const int32_t* ci,
                                                              int advance, const uint8_t* force,
                                                              int32_t* slot_wp, int32_t* row_wp,
                                                              uint8_t* row_flush, int32_t* dev_err) {
    extern __shared__ __align__(16) float psm[];
    __shared__ int sh_w;
    const int b = blockIdx.x;
    const int s = ci[b];
    if (threadIdx.x == 0)
        sh_w = advance ? standard_cursor(b, s, a.num_slots, a.L, slot_wp, force, row_wp, row_flush,
                                         dev_err)
                       : given_cursor(b, s, a.num_slots, a.L, row_wp, dev_err);
    if (s >= 0 && s < a.num_slots) stage_slot(a, b, s, psm);
    __syncthreads();
    const int w = sh_w;
    if (w < 0) return;
    append_row(a, b, s, w);
    const int H = a.H, N = a.N, G = a.G, L = a.L;
    const int sa = a.act_bf16 ? 2 : 4;
    float* dts = psm + G * N;
    for (int h = threadIdx.x; h < H; h += blockDim.x) dts[h * (L + 1) + w] = step_dt(a, b, h);
    char* braw = reinterpret_cast<char*>(psm + ((G * N + H * (L + 1) + G * L + 3) & ~3));
    const int bcn = N * sa / 16;
    for (int c = threadIdx.x; c < G * bcn; c += blockDim.x) {
        const int g = c / bcn, j = c - (c / bcn) * bcn;
        reinterpret_cast<uint4*>(braw + ((size_t)g * L + w) * N * sa)[j] =
            reinterpret_cast<const uint4*>(static_cast<const char*>(a.B) + (size_t)b * G * N * sa)[c];
    }
    __syncthreads();
    tables_from_smem(a, b, w, psm);
}

RowArgs row_args(const rssm_mamba2_dims* d) {
    RowArgs a{};
    a.H = d->nheads;
    a.P = d->headdim;
    a.N = d->dstate;
    a.G = d->ngroups;
    a.L = d->ring_len;
    a.num_slots = d->num_slots;
    a.act_bf16 = d->act_dtype == RSSM_BF16;
    return a;
}

}  // namespace m2
}  // namespace rssm

using namespace rssm;

extern "C" int rssm_ring_append(const rssm_mamba2_dims* d, const void* x, const float* dt_raw,
                                const float* dt_bias, int dt_softplus, const void* B,
                                const int32_t* cache_indices, const int32_t* row_wp, void* ring_x,
                                float* ring_dt, void* ring_B, int32_t* dev_err,
                                rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(x) || !ok_ptr(dt_raw) || !ok_opt_ptr(dt_bias) || !ok_ptr(B) ||
        !ok_ptr(cache_indices) || !ok_ptr(row_wp) || !ok_ptr(ring_x) || !ok_ptr(ring_dt) ||
        !ok_ptr(ring_B))
        return RSSM_ERR_INVALID_ARG;
    m2::RowArgs ra = m2::row_args(d);
    ra.x = x;
    ra.dt_raw = dt_raw;
    ra.dt_bias = dt_bias;
    ra.softplus = dt_softplus;
    ra.B = B;
    ra.ring_x = ring_x;
    ra.ring_dt = ring_dt;
    ra.ring_B = ring_B;
    m2::ring_append_kernel<<<d->batch, 256, 0, (cudaStream_t)stream>>>(ra, cache_indices, row_wp,
                                                                       dev_err);
    return launch_status();
}

extern "C" size_t rssm_mamba2_workspace_size(const rssm_mamba2_dims* d) {
    if (m2::check_dims(d)) return 0;
    return (size_t)d->batch * d->nheads * m2::tbl_floats(d->ring_len) * sizeof(float);
}

// Shared-memory size of the table-building kernels, checked and opted in.
static int m2_prologue_smem(const rssm_mamba2_dims* d, const void* kernel, int* smem) {
    *smem = m2::prologue_smem(d->nheads, d->dstate, d->ngroups, d->ring_len,
                              d->act_dtype == RSSM_BF16 ? 2 : 4);
    DeviceInfo di;
    if (!device_info(&di)) return RSSM_ERR_CUDA;
    if (*smem > di.max_smem_optin) return RSSM_ERR_UNSUPPORTED;
    if (*smem > 48 * 1024 && !ensure_smem_limit(kernel, *smem)) return RSSM_ERR_CUDA;
    return RSSM_OK;
}

extern "C" int rssm_mamba2_precompute(const rssm_mamba2_dims* d, const float* A, const void* C,
                                      const float* ring_dt, const void* ring_B,
                                      const int32_t* cache_indices, const int32_t* row_wp,
                                      void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                      rssm_stream_t stream) {
    (void)dev_err;
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(A) || !ok_ptr(C) || !ok_ptr(ring_dt) || !ok_ptr(ring_B) || !ok_ptr(cache_indices) ||
        !ok_ptr(row_wp) || !ok_ptr(workspace))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_mamba2_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    int smem = 0;
    rc = m2_prologue_smem(d, reinterpret_cast<const void*>(m2::precompute_kernel), &smem);
    if (rc) return rc;
    m2::RowArgs ra = m2::row_args(d);
    ra.A = A;
    ra.C = C;
    ra.ring_dt = const_cast<float*>(ring_dt);  // read only here
    ra.ring_B = const_cast<void*>(ring_B);
    ra.ws = static_cast<float*>(workspace);
    m2::precompute_kernel<<<d->batch, m2::kRowThreads, smem, (cudaStream_t)stream>>>(ra, cache_indices, row_wp);
    return launch_status();
}

extern "C" int rssm_mamba2_prepare(const rssm_mamba2_dims* d, int advance,
                                   const uint8_t* force_flush, int32_t* slot_wp, int32_t* row_wp,
                                   uint8_t* row_flush, const void* x, const float* dt_raw,
                                   const float* dt_bias, int dt_softplus, const void* B,
                                   const float* A, const void* C, const int32_t* cache_indices,
                                   void* ring_x, float* ring_dt, void* ring_B, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_err,
                                   rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(row_wp) || (advance && (!ok_ptr(slot_wp) || !ok_ptr(row_flush))) ||
        !ok_opt_ptr(force_flush) || !ok_ptr(x) || !ok_ptr(dt_raw) || !ok_opt_ptr(dt_bias) ||
        !ok_ptr(B) || !ok_ptr(A) || !ok_ptr(C) || !ok_ptr(cache_indices) || !ok_ptr(ring_x) ||
        !ok_ptr(ring_dt) || !ok_ptr(ring_B) || !ok_ptr(workspace))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_mamba2_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    int smem = 0;
    m2::RowArgs ra = m2::row_args(d);
    ra.x = x;
    ra.dt_raw = dt_raw;
    ra.dt_bias = dt_bias;
    ra.softplus = dt_softplus;
    ra.B = B;
    ra.A = A;
    ra.C = C;
    ra.ring_x = ring_x;
    ra.ring_dt = ring_dt;
    ra.ring_B = ring_B;
    ra.ws = static_cast<float*>(workspace);
    rc = m2_prologue_smem(d, reinterpret_cast<const void*>(m2::prepare_kernel), &smem);
    if (rc) return rc;
    m2::prepare_kernel<<<d->batch, m2::kRowThreads, smem, (cudaStream_t)stream>>>(
        ra, cache_indices, advance ? 1 : 0, force_flush, slot_wp, row_wp, row_flush, dev_err);
    return launch_status();
}
