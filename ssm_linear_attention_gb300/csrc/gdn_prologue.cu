// gdn_prologue.cu -- the per-row prologue of a gated-delta-net ReplaySSM decode
// step on sm_103a: ring append (k, g), coefficient tables, and both fused with
// the cursor step in one launch.
//
// Pages followed: [GDN] "GDN ReplaySSM decode (Part A of RFC 28511)" (SGLang PR
// 28451 report): 实现拆解 item 1 (non-flush outputs reconstructed from the
// checkpoint and the ring, which needs the key dot products and gate products
// per row), 实现拆解 item 2 (per-row cursors with a forced-flush mask), 实现拆解
// item 3 (the k and g rings).
//
// Kernels (one CTA per row):
//   ring_append_kernel  k, g into ring entry w (128 threads).
//   precompute_kernel   warp per key head: k_i . k_t, k_i . q_t for ring entries
//                       i < w, k_t . q_t; then gate products per value head into
//                       per-(row, value head) tables (512 threads).
//   prepare_kernel      cursor step + ring append + tables in one CTA.
#include "common.cuh"
#include "cursor.cuh"
#include "gdn.cuh"
#include "internal.h"

namespace rssm {
namespace gdn {

// ----------------------------------------------------------------------------
// per-row prologue pieces: ring append (k, g), coefficient tables
// ----------------------------------------------------------------------------

struct RowArgs {
    int HV, HK, L, num_slots, act_bf16;
    const void* q;       // [batch][HK][K]
    const void* k;       // [batch][HK][K]
    const float* beta;   // [batch][HV]
    const float* g;      // [batch][HV]
    void* ring_k;        // [slots][HK][L][K]
    float* ring_g;       // [slots][HV][L]
    float* ws;           // [batch][HV][TBL]
};

// Entry w of slot s's rings <- row b's k (key heads [k0, k1)) and g (their value
// heads).
__device__ void append_heads(const RowArgs& a, int b, int s, int w, int k0, int k1) {
    const int HV = a.HV, HK = a.HK, L = a.L, vpk = HV / HK;
    const int sa = a.act_bf16 ? 2 : 4;
    const int kc = KD * sa / 16;
    const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const char*>(a.k) +
                                                     ((size_t)b * HK + k0) * KD * sa);
    for (int c = threadIdx.x; c < (k1 - k0) * kc; c += blockDim.x) {
        const int kh = k0 + c / kc, j = c % kc;
        reinterpret_cast<uint4*>(static_cast<char*>(a.ring_k) +
                                 (((size_t)s * HK + kh) * L + w) * KD * sa)[j] = ks[c];
    }
    for (int hv = k0 * vpk + threadIdx.x; hv < k1 * vpk; hv += blockDim.x)
        a.ring_g[((size_t)s * HV + hv) * L + w] = a.g[(size_t)b * HV + hv];
}

// Shared memory of precompute_heads for nk key heads and nv value heads, in bytes.
__host__ __device__ inline int precompute_smem(int nv, int nk, int L) {
    return (((2 * nk * L + nk + 3) & ~3) + nv * tbl_floats(L) + nv * L) * 4;
}

// Row b's tables for the key heads [k0, k1) and their value heads, from ring
// entries 0..w-1 (k, g) and the step's q, k, beta, g. A warp per key head: lanes
// hold 4 key columns of k_t and q_t, and each ring key k_i (i < w) is read with
// one coalesced warp load; the two dot products reduce with a butterfly. Then per
// value head (key head kh = hv / (HV/HK)):
//   gamma_i = prod_{j=i+1..w-1} g_j, Gamma_i = g_t gamma_i,
//   t[i] = gamma_i (k_i . k_t), t[L+i] = Gamma_i (k_i . q_t), t[2L+i] = Gamma_i
//   (Gamma_w = 1), Gu = gamma_{-1}, Go = g_t Gu, k_t . q_t, beta_t, g_t.
// The ring entries read are never the one appended this step, so the fused
// kernels need no ordering between the append and these loads.
__device__ void precompute_heads(const RowArgs& a, int b, int s, int w, int k0, int k1,
                                 float* psm) {
    const int HV = a.HV, HK = a.HK, L = a.L, vpk = HV / HK;
    const int nk = k1 - k0, nv = nk * vpk, v0 = k0 * vpk;
    const int TBL = tbl_floats(L);
    const bool bf = a.act_bf16;
    const int sa = bf ? 2 : 4;
    float* kk = psm;            // [nk][L]
    float* kq = kk + nk * L;    // [nk][L]
    float* kqt = kq + nk * L;   // [nk]
    float* tbl = psm + ((2 * nk * L + nk + 3) & ~3);  // [nv][TBL]
    float* gs = tbl + nv * TBL;                        // gate ring [nv][L]

    for (int e = threadIdx.x; e < nv * w; e += blockDim.x) {
        const int hl = e / w, i = e - (e / w) * w;
        gs[hl * L + i] = a.ring_g[((size_t)s * HV + v0 + hl) * L + i];
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int kl = warp; kl < nk; kl += nwarps) {
        const int kh = k0 + kl;
        float kt[4], qt[4];
        load4(static_cast<const char*>(a.k) + ((size_t)b * HK + kh) * KD * sa, lane * 4, bf, kt);
        load4(static_cast<const char*>(a.q) + ((size_t)b * HK + kh) * KD * sa, lane * 4, bf, qt);
        const char* kr = static_cast<const char*>(a.ring_k) + ((size_t)s * HK + kh) * L * KD * sa;
        float t0 = kt[0] * qt[0] + kt[1] * qt[1] + kt[2] * qt[2] + kt[3] * qt[3];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) t0 += __shfl_xor_sync(0xffffffffu, t0, o);
        if (lane == 0) kqt[kl] = t0;
        for (int i0 = 0; i0 < w; i0 += 4) {
            float ki[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (i0 + u < w) load4(kr + (size_t)(i0 + u) * KD * sa, lane * 4, bf, ki[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (i0 + u < w) {
                    float d1 = ki[u][0] * kt[0] + ki[u][1] * kt[1] + ki[u][2] * kt[2] + ki[u][3] * kt[3];
                    float d2 = ki[u][0] * qt[0] + ki[u][1] * qt[1] + ki[u][2] * qt[2] + ki[u][3] * qt[3];
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) {
                        d1 += __shfl_xor_sync(0xffffffffu, d1, o);
                        d2 += __shfl_xor_sync(0xffffffffu, d2, o);
                    }
                    if (lane == 0) {
                        kk[kl * L + i0 + u] = d1;
                        kq[kl * L + i0 + u] = d2;
                    }
                }
            }
        }
    }
    __syncthreads();
    for (int hl = threadIdx.x; hl < nv; hl += blockDim.x) {
        const int hv = v0 + hl, kl = hl / vpk;
        const float gt = a.g[(size_t)b * HV + hv];
        const float bt = a.beta[(size_t)b * HV + hv];
        const float* gr = gs + hl * L;
        float* t = tbl + hl * TBL;
        float gam = 1.f;  // prod_{j=i+1..w-1} g_j
        for (int i = w - 1; i >= 0; --i) {
            const float Gi = gt * gam;
            t[i] = gam * kk[kl * L + i];
            t[L + i] = Gi * kq[kl * L + i];
            t[2 * L + i] = Gi;
            gam *= gr[i];
        }
        for (int i = w; i < L; ++i) {
            t[i] = 0.f;
            t[L + i] = 0.f;
            t[2 * L + i] = (i == w) ? 1.f : 0.f;
        }
        t[3 * L] = gam;
        t[3 * L + 1] = gt * gam;
        t[3 * L + 2] = kqt[kl];
        t[3 * L + 3] = bt;
        t[3 * L + 4] = gt;
        for (int i = 3 * L + 5; i < TBL; ++i) t[i] = 0.f;
    }
    __syncthreads();
    float4* dst = reinterpret_cast<float4*>(a.ws + ((size_t)b * HV + v0) * TBL);
    const float4* src = reinterpret_cast<const float4*>(tbl);
    for (int c = threadIdx.x; c < nv * TBL / 4; c += blockDim.x) dst[c] = src[c];
}

// ----------------------------------------------------------------------------
// prologue kernels
// ----------------------------------------------------------------------------

__global__ void __launch_bounds__(128) ring_append_kernel(const RowArgs a, const int32_t* ci,
                                                          const int32_t* row_wp, int32_t* dev_err) {
    const int b = blockIdx.x;
    const int w = given_cursor(b, ci[b], a.num_slots, a.L, row_wp, threadIdx.x == 0 ? dev_err : nullptr);
    if (w < 0) return;
    append_heads(a, b, ci[b], w, 0, a.HK);
}

__global__ void __launch_bounds__(512) precompute_kernel(const RowArgs a, const int32_t* ci,
                                                         const int32_t* row_wp) {
    extern __shared__ __align__(16) float psm[];
    const int b = blockIdx.x;
    // bad slots and cursors are reported by the append and output kernels
    const int w = given_cursor(b, ci[b], a.num_slots, a.L, row_wp, nullptr);
    if (w < 0) return;
    precompute_heads(a, b, ci[b], w, 0, a.HK, psm);
}

// Cursor advance (when `advance`), ring append and tables of one row in one CTA.
__global__ void __launch_bounds__(512) prepare_kernel(const RowArgs a, const int32_t* ci,
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
    append_heads(a, b, s, w, 0, a.HK);
    precompute_heads(a, b, s, w, 0, a.HK, psm);
}

RowArgs row_args(const rssm_gdn_dims* d) {
    RowArgs a{};
    a.HV = d->num_v_heads;
    a.HK = d->num_k_heads;
    a.L = d->ring_len;
    a.num_slots = d->num_slots;
    a.act_bf16 = d->act_dtype == RSSM_BF16;
    return a;
}

}  // namespace gdn
}  // namespace rssm

using namespace rssm;

extern "C" int rssm_gdn_ring_append(const rssm_gdn_dims* d, const void* k, const float* g,
                                    const int32_t* cache_indices, const int32_t* row_wp,
                                    void* ring_k, float* ring_g, int32_t* dev_err,
                                    rssm_stream_t stream) {
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(k) || !ok_ptr(g) || !ok_ptr(cache_indices) || !ok_ptr(row_wp) || !ok_ptr(ring_k) ||
        !ok_ptr(ring_g))
        return RSSM_ERR_INVALID_ARG;
    gdn::RowArgs ra = gdn::row_args(d);
    ra.k = k;
    ra.g = g;
    ra.ring_k = ring_k;
    ra.ring_g = ring_g;
    gdn::ring_append_kernel<<<d->batch, 128, 0, (cudaStream_t)stream>>>(ra, cache_indices, row_wp,
                                                                        dev_err);
    return launch_status();
}

extern "C" size_t rssm_gdn_workspace_size(const rssm_gdn_dims* d) {
    if (gdn::check_dims(d)) return 0;
    return (size_t)d->batch * d->num_v_heads * gdn::tbl_floats(d->ring_len) * sizeof(float);
}

// Shared-memory size of the table-building kernels, checked and opted in.
static int gdn_prologue_smem(const rssm_gdn_dims* d, const void* kernel, int key_heads, int* smem) {
    *smem = gdn::precompute_smem(key_heads * (d->num_v_heads / d->num_k_heads), key_heads,
                                 d->ring_len);
    DeviceInfo di;
    if (!device_info(&di)) return RSSM_ERR_CUDA;
    if (*smem > di.max_smem_optin) return RSSM_ERR_UNSUPPORTED;
    if (*smem > 48 * 1024 && !ensure_smem_limit(kernel, *smem)) return RSSM_ERR_CUDA;
    return RSSM_OK;
}

extern "C" int rssm_gdn_precompute(const rssm_gdn_dims* d, const void* q, const void* k,
                                   const float* beta, const float* g, const void* ring_k,
                                   const float* ring_g, const int32_t* cache_indices,
                                   const int32_t* row_wp, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_err, rssm_stream_t stream) {
    (void)dev_err;
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(beta) || !ok_ptr(g) || !ok_ptr(ring_k) ||
        !ok_ptr(ring_g) || !ok_ptr(cache_indices) || !ok_ptr(row_wp) || !ok_ptr(workspace))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_gdn_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    int smem = 0;
    rc = gdn_prologue_smem(d, reinterpret_cast<const void*>(gdn::precompute_kernel), d->num_k_heads, &smem);
    if (rc) return rc;
    gdn::RowArgs ra = gdn::row_args(d);
    ra.q = q;
    ra.k = k;
    ra.beta = beta;
    ra.g = g;
    ra.ring_k = const_cast<void*>(ring_k);  // read only here
    ra.ring_g = const_cast<float*>(ring_g);
    ra.ws = static_cast<float*>(workspace);
    gdn::precompute_kernel<<<d->batch, 512, smem, (cudaStream_t)stream>>>(ra, cache_indices, row_wp);
    return launch_status();
}

extern "C" int rssm_gdn_prepare(const rssm_gdn_dims* d, int advance, const uint8_t* force_flush,
                                int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush,
                                const void* q, const void* k, const float* beta, const float* g,
                                const int32_t* cache_indices, void* ring_k, float* ring_g,
                                void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                rssm_stream_t stream) {
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(row_wp) || (advance && (!ok_ptr(slot_wp) || !ok_ptr(row_flush))) ||
        !ok_opt_ptr(force_flush) || !ok_ptr(q) || !ok_ptr(k) || !ok_ptr(beta) || !ok_ptr(g) ||
        !ok_ptr(cache_indices) || !ok_ptr(ring_k) || !ok_ptr(ring_g) || !ok_ptr(workspace))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_gdn_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    int smem = 0;
    gdn::RowArgs ra = gdn::row_args(d);
    ra.q = q;
    ra.k = k;
    ra.beta = beta;
    ra.g = g;
    ra.ring_k = ring_k;
    ra.ring_g = ring_g;
    ra.ws = static_cast<float*>(workspace);
    const int adv = advance ? 1 : 0;
    rc = gdn_prologue_smem(d, reinterpret_cast<const void*>(gdn::prepare_kernel), d->num_k_heads,
                           &smem);
    if (rc) return rc;
    gdn::prepare_kernel<<<d->batch, 512, smem, (cudaStream_t)stream>>>(
        ra, cache_indices, adv, force_flush, slot_wp, row_wp, row_flush, dev_err);
    return launch_status();
}
