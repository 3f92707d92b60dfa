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
// Kernels (one CTA of 256 threads per row):
//   ring_append_kernel  x, dt = softplus(dt_raw + dt_bias), B into ring entry w.
//   precompute_kernel   B_i . C_t per group from the staged B run, decay suffix
//                       products per head, written as per-(row, head) tables.
//   prepare_kernel      cursor step + ring append + tables in one CTA.
#include "common.cuh"
#include "cursor.cuh"
#include "internal.h"
#include "mamba2.cuh"

namespace rssm {
namespace m2 {

// ----------------------------------------------------------------------------
// per-row prologue pieces: ring append, coefficient tables
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

// Entry w of slot s's rings <- row b's x, dt = softplus(dt_raw + dt_bias), B, for
// the groups [g0, g1) and their heads.
__device__ void append_groups(const RowArgs& a, int b, int s, int w, int g0, int g1) {
    const int H = a.H, P = a.P, N = a.N, G = a.G, L = a.L;
    const int hpg = H / G, h0 = g0 * hpg, nh = (g1 - g0) * hpg;
    const int sa = a.act_bf16 ? 2 : 4;
    const int xc = P * sa / 16;  // 16-byte chunks per head row
    const uint4* xs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.x) +
                                                     ((size_t)b * H + h0) * P * sa);
    for (int c = threadIdx.x; c < nh * xc; c += blockDim.x) {
        const int h = h0 + c / xc, j = c % xc;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(a.ring_x) +
                                              (((size_t)s * H + h) * L + w) * P * sa) + j;
        *dst = xs[c];
    }
    for (int hl = threadIdx.x; hl < nh; hl += blockDim.x) {
        const int h = h0 + hl;
        float v = a.dt_raw[(size_t)b * H + h] + (a.dt_bias ? a.dt_bias[h] : 0.f);
        if (a.softplus) v = softplus_f(v);
        a.ring_dt[((size_t)s * H + h) * L + w] = v;
    }
    const int bc = N * sa / 16;
    const uint4* bs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.B) +
                                                     ((size_t)b * G + g0) * N * sa);
    for (int c = threadIdx.x; c < (g1 - g0) * bc; c += blockDim.x) {
        const int g = g0 + c / bc, j = c % bc;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(a.ring_B) +
                                              (((size_t)s * G + g) * L + w) * N * sa) + j;
        *dst = bs[c];
    }
}

// Shared memory of precompute_groups for ng groups of hpg heads, in bytes.
__host__ __device__ inline int precompute_smem(int nh, int N, int ng, int L, int sa) {
    return (((ng * N + nh * L + ng * L + 3) & ~3) + nh * tbl_floats(L)) * 4 + ng * L * N * sa;
}

// Row b's tables for the groups [g0, g1) from ring entries 0..w (read with
// L2-coherent loads, so entries this block appended just before are seen):
//   P_i = exp(A_h sum_{j>i} dt_j), coef_i = P_i dt_i (B_i . C_t), a_i = P_i dt_i,
//   Pm1 = exp(A_h sum_{j<=w} dt_j).
__device__ void precompute_groups(const RowArgs& a, int b, int s, int w, int g0, int g1,
                                  float* psm) {
    const int H = a.H, N = a.N, G = a.G, L = a.L;
    const int TBL = tbl_floats(L);
    const bool bf = a.act_bf16;
    const int sa = bf ? 2 : 4;
    const int hpg = H / G, ng = g1 - g0, nh = ng * hpg, h0 = g0 * hpg;
    float* cs = psm;                                           // [ng][N] C_t in fp32
    float* dts = cs + ng * N;                                  // [nh][L] dt of entries 0..w
    float* bc = dts + nh * L;                                  // [ng][L] B_i . C_t
    float* tbl = psm + ((ng * N + nh * L + ng * L + 3) & ~3);  // [nh][TBL]
    char* braw = reinterpret_cast<char*>(tbl + nh * TBL);      // [ng][w+1][N] raw B entries

    // stage C_t, the dt run and the B run of every group with coalesced loads
    for (int e = threadIdx.x * 8; e < ng * N; e += blockDim.x * 8)
        load8(static_cast<const char*>(a.C) + (((size_t)b * G + g0) * N + e) * sa, bf, cs + e);
    for (int e = threadIdx.x; e < nh * (w + 1); e += blockDim.x) {
        const int hl = e / (w + 1), i = e - (e / (w + 1)) * (w + 1);
        dts[hl * L + i] = __ldcg(a.ring_dt + ((size_t)s * H + h0 + hl) * L + i);
    }
    const int run16 = (w + 1) * N * sa / 16;  // 16-byte chunks of one group's run
    for (int e = threadIdx.x; e < ng * run16; e += blockDim.x) {
        const int gl = e / run16, c = e - (e / run16) * run16;
        reinterpret_cast<uint4*>(braw)[e] = __ldcg(reinterpret_cast<const uint4*>(
            static_cast<const char*>(a.ring_B) + ((size_t)s * G + g0 + gl) * L * N * sa) + c);
    }
    __syncthreads();

    // bc[g][i] = B_i . C_t: one warp per (group, entry), lanes over dstate
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int pair = warp; pair < ng * (w + 1); pair += nwarps) {
        const int gl = pair / (w + 1), i = pair - (pair / (w + 1)) * (w + 1);
        const char* Bi = braw + (size_t)(gl * (w + 1) + i) * N * sa;
        const float* cg = cs + gl * N;
        float acc = 0.f;
        for (int n = lane; n < N; n += 32) acc = fmaf(load1(Bi, n, bf), cg[n], acc);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) bc[gl * L + i] = acc;
    }
    __syncthreads();

    for (int hl = threadIdx.x; hl < nh; hl += blockDim.x) {
        const int gl = hl / hpg;
        const float* dh = dts + hl * L;
        float* t = tbl + hl * TBL;
        const float Ah = a.A[h0 + hl];
        float suffix = 0.f;
        for (int i = w; i >= 0; --i) {
            const float dti = dh[i];
            const float Pi = expf(Ah * suffix);
            t[i] = Pi * dti * bc[gl * L + i];
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
    __syncthreads();
    float4* dst = reinterpret_cast<float4*>(a.ws + ((size_t)b * H + h0) * TBL);
    const float4* src = reinterpret_cast<const float4*>(tbl);
    for (int c = threadIdx.x; c < nh * TBL / 4; c += blockDim.x) dst[c] = src[c];
}

// ----------------------------------------------------------------------------
// prologue kernels
// ----------------------------------------------------------------------------

__global__ void __launch_bounds__(256) ring_append_kernel(const RowArgs a, const int32_t* ci,
                                                          const int32_t* row_wp, int32_t* dev_err) {
    const int b = blockIdx.x;
    const int w = given_cursor(b, ci[b], a.num_slots, a.L, row_wp, threadIdx.x == 0 ? dev_err : nullptr);
    if (w < 0) return;
    append_groups(a, b, ci[b], w, 0, a.G);
}

__global__ void __launch_bounds__(256) precompute_kernel(const RowArgs a, const int32_t* ci,
                                                         const int32_t* row_wp) {
    extern __shared__ __align__(16) float psm[];
    const int b = blockIdx.x;
    // bad slots and cursors are reported by the append and output kernels
    const int w = given_cursor(b, ci[b], a.num_slots, a.L, row_wp, nullptr);
    if (w < 0) return;
    precompute_groups(a, b, ci[b], w, 0, a.G, psm);
}

// Cursor advance (when `advance`), ring append and tables of one row in one CTA.
__global__ void __launch_bounds__(256) prepare_kernel(const RowArgs a, const int32_t* ci,
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
    __syncthreads();
    const int w = sh_w;
    if (w < 0) return;
    append_groups(a, b, s, w, 0, a.G);
    __syncthreads();  // the appended entry is visible to the whole block
    precompute_groups(a, b, s, w, 0, a.G, psm);
}

// The same with one CTA per (row, group), the G CTAs of a row forming a thread-
// block cluster: every CTA reads the slot's cursor, the cluster barrier orders
// those reads before the cluster's first CTA advances it, and each CTA appends
// and builds the tables of its own group.
__global__ void __launch_bounds__(128) prepare_cluster_kernel(const RowArgs a, const int32_t* ci,
                                                              int advance, const uint8_t* force,
                                                              int32_t* slot_wp, int32_t* row_wp,
                                                              uint8_t* row_flush, int32_t* dev_err) {
    extern __shared__ __align__(16) float psm[];
    __shared__ int sh_w;
    const int b = blockIdx.x / a.G, g = blockIdx.x - (blockIdx.x / a.G) * a.G;
    const int s = ci[b];
    if (threadIdx.x == 0) {
        int w = -1;
        if (s >= 0 && s < a.num_slots) {
            w = advance ? slot_wp[s] : row_wp[b];
            if (w < 0 || w >= a.L) {
                if (g == 0) set_dev_err(dev_err, RSSM_DEVERR_CURSOR);
                w = -1;
            }
        } else if (s >= a.num_slots && g == 0) {
            set_dev_err(dev_err, RSSM_DEVERR_SLOT);
        }
        sh_w = w;
    }
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
    const int w = sh_w;
    if (advance && g == 0 && threadIdx.x == 0) {
        const int f = w >= 0 && ((w == a.L - 1) || (force != nullptr && force[b] != 0));
        row_wp[b] = w >= 0 ? w : 0;
        row_flush[b] = static_cast<uint8_t>(f);
        if (w >= 0) slot_wp[s] = f ? 0 : w + 1;
    }
    if (w < 0) return;
    append_groups(a, b, s, w, g, g + 1);
    __syncthreads();  // the appended entries are visible to the whole block
    precompute_groups(a, b, s, w, g, g + 1, psm);
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
static int m2_prologue_smem(const rssm_mamba2_dims* d, const void* kernel, int groups, int* smem) {
    *smem = m2::precompute_smem(groups * (d->nheads / d->ngroups), d->dstate, groups, d->ring_len,
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
    rc = m2_prologue_smem(d, reinterpret_cast<const void*>(m2::precompute_kernel), d->ngroups, &smem);
    if (rc) return rc;
    m2::RowArgs ra = m2::row_args(d);
    ra.A = A;
    ra.C = C;
    ra.ring_dt = const_cast<float*>(ring_dt);  // read only here
    ra.ring_B = const_cast<void*>(ring_B);
    ra.ws = static_cast<float*>(workspace);
    m2::precompute_kernel<<<d->batch, 256, smem, (cudaStream_t)stream>>>(ra, cache_indices, row_wp);
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
    const int adv = advance ? 1 : 0;
    if (d->ngroups <= 8) {
        // one CTA per (row, group); the row's CTAs form a cluster
        rc = m2_prologue_smem(d, reinterpret_cast<const void*>(m2::prepare_cluster_kernel), 1, &smem);
        if (rc) return rc;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)d->batch * d->ngroups);
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = (cudaStream_t)stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = d->ngroups;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, m2::prepare_cluster_kernel, ra, cache_indices, adv, force_flush,
                               slot_wp, row_wp, row_flush, dev_err) != cudaSuccess) {
            cudaGetLastError();
            return RSSM_ERR_CUDA;
        }
        return launch_status();
    }
    rc = m2_prologue_smem(d, reinterpret_cast<const void*>(m2::prepare_kernel), d->ngroups, &smem);
    if (rc) return rc;
    m2::prepare_kernel<<<d->batch, 256, smem, (cudaStream_t)stream>>>(
        ra, cache_indices, adv, force_flush, slot_wp, row_wp, row_flush, dev_err);
    return launch_status();
}
