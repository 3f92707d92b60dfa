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
//   precompute_kernel   stages the step's q, k, beta, g and the slot's k and g
//                       rings with 1-D bulk copies on one mbarrier; k_i . k_t and
//                       k_i . q_t (eight lanes per entry), k_t . q_t; gate products
//                       per value head by a segmented warp scan; tables written
//                       straight to the workspace (512 threads).
//   prepare_kernel      cursor step + ring append + tables: the staging copies are
//                       issued before the cursor is read.
#include "common.cuh"
#include "cursor.cuh"
#include "gdn.cuh"
#include "internal.h"

namespace rssm {
namespace gdn {

// ----------------------------------------------------------------------------
// per-row prologue pieces
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

constexpr int kRowThreads = 512;

// Entry w of slot s's rings <- row b's k and g.
__device__ void append_row(const RowArgs& a, int b, int s, int w) {
    const int HV = a.HV, HK = a.HK, L = a.L;
    const int sa = a.act_bf16 ? 2 : 4;
    const int kc = KD * sa / 16;
    const uint4* ks =
        reinterpret_cast<const uint4*>(static_cast<const char*>(a.k) + (size_t)b * HK * KD * sa);
    for (int c = threadIdx.x; c < HK * kc; c += blockDim.x) {
        const int kh = c / kc, j = c % kc;
        reinterpret_cast<uint4*>(static_cast<char*>(a.ring_k) +
                                 (((size_t)s * HK + kh) * L + w) * KD * sa)[j] = ks[c];
    }
    for (int hv = threadIdx.x; hv < HV; hv += blockDim.x)
        a.ring_g[((size_t)s * HV + hv) * L + w] = a.g[(size_t)b * HV + hv];
}

// Shared memory of the table-building kernels (byte offsets, 16-byte aligned): the
// step's k_t, q_t [HK][K] (activation type), the slot's k ring [HK][L][K]
// (activation type), its g ring [HV][L], beta_t, g_t [HV], k_i . k_t and k_i . q_t
// [HK][L], k_t . q_t [HK] (fp32).
struct ProLayout {
    int kt, qt, kr, gr, bt, gt, kk, kq, kqt, total;
    __host__ __device__ ProLayout(int HV, int HK, int L, int sa) {
        auto up = [](int x) { return (x + 15) & ~15; };
        kt = 0;
        qt = kt + up(HK * KD * sa);
        kr = qt + up(HK * KD * sa);
        gr = kr + up(HK * L * KD * sa);
        bt = gr + up(HV * L * 4);
        gt = bt + up(HV * 4);
        kk = gt + up(HV * 4);
        kq = kk + up(HK * L * 4);
        kqt = kq + up(HK * L * 4);
        total = kqt + up(HK * 4);
    }
};

// Stage row b's k_t, q_t, beta_t, g_t and slot s's k and g rings with 1-D bulk
// copies completing on `bar` (issued by one thread; the fp32 per-head vectors fall
// back to plain loads when their sizes are not multiples of 16 bytes).
__device__ void stage_issue(const RowArgs& a, int b, int s, uint8_t* sm, uint64_t* bar) {
    const int HV = a.HV, HK = a.HK, L = a.L;
    const int sa = a.act_bf16 ? 2 : 4;
    const ProLayout lo(HV, HK, L, sa);
    const bool bulk_v = (HV & 3) == 0 && ((HV * L) & 3) == 0;
    const uint32_t kb = HK * KD * sa;
    mbar_arrive_expect_tx(bar, 2 * kb + HK * L * KD * sa + (bulk_v ? (HV * L + 2 * HV) * 4 : 0));
    bulk_g2s(sm + lo.kt, static_cast<const char*>(a.k) + (size_t)b * kb, kb, bar);
    bulk_g2s(sm + lo.qt, static_cast<const char*>(a.q) + (size_t)b * kb, kb, bar);
    bulk_g2s(sm + lo.kr, static_cast<const char*>(a.ring_k) + (size_t)s * HK * L * KD * sa,
             HK * L * KD * sa, bar);
    if (bulk_v) {
        bulk_g2s(sm + lo.gr, a.ring_g + (size_t)s * HV * L, HV * L * 4, bar);
        bulk_g2s(sm + lo.bt, a.beta + (size_t)b * HV, HV * 4, bar);
        bulk_g2s(sm + lo.gt, a.g + (size_t)b * HV, HV * 4, bar);
    } else {
        float* gr = reinterpret_cast<float*>(sm + lo.gr);
        float* bt = reinterpret_cast<float*>(sm + lo.bt);
        float* gt = reinterpret_cast<float*>(sm + lo.gt);
        for (int i = 0; i < HV * L; ++i) gr[i] = a.ring_g[(size_t)s * HV * L + i];
        for (int h = 0; h < HV; ++h) {
            bt[h] = a.beta[(size_t)b * HV + h];
            gt[h] = a.g[(size_t)b * HV + h];
        }
    }
}

// Row b's tables from the staged data, ring entries 0..w-1 and the step:
//   gamma_i = prod_{j=i+1..w-1} g_j, Gamma_i = g_t gamma_i,
//   t[i] = gamma_i (k_i . k_t), t[L+i] = Gamma_i (k_i . q_t), t[2L+i] = Gamma_i
//   (Gamma_w = 1), Gu = gamma_{-1}, Go = g_t Gu, k_t . q_t, beta_t, g_t.
// Dots: a warp per key head, eight lanes per entry (K/8 columns each). Gate
// products: a segment of LS = pow2ceil(L) <= 32 lanes per value head, lane i =
// entry i, by a segmented product scan.
__device__ void tables_from_smem(const RowArgs& a, int b, int w, uint8_t* sm) {
    const int HV = a.HV, HK = a.HK, L = a.L, vpk = HV / HK;
    const int TBL = tbl_floats(L);
    const bool bf = a.act_bf16;
    const int sa = bf ? 2 : 4;
    const ProLayout lo(HV, HK, L, sa);
    const char* kt = reinterpret_cast<const char*>(sm + lo.kt);
    const char* qt = reinterpret_cast<const char*>(sm + lo.qt);
    const char* kr = reinterpret_cast<const char*>(sm + lo.kr);
    const float* gr = reinterpret_cast<const float*>(sm + lo.gr);
    const float* bt = reinterpret_cast<const float*>(sm + lo.bt);
    const float* gt = reinterpret_cast<const float*>(sm + lo.gt);
    float* kk = reinterpret_cast<float*>(sm + lo.kk);
    float* kq = reinterpret_cast<float*>(sm + lo.kq);
    float* kqt = reinterpret_cast<float*>(sm + lo.kqt);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int sub = lane >> 3, part = lane & 7;
    constexpr int per = KD / 8;
    for (int kh = warp; kh < HK; kh += nwarps) {
        float ktv[per], qtv[per];
        load8(kt + ((size_t)kh * KD + part * per) * sa, bf, ktv);
        load8(kt + ((size_t)kh * KD + part * per + 8) * sa, bf, ktv + 8);
        load8(qt + ((size_t)kh * KD + part * per) * sa, bf, qtv);
        load8(qt + ((size_t)kh * KD + part * per + 8) * sa, bf, qtv + 8);
        // entries w.. are unused; slot w of the pass computes k_t . q_t
        for (int i0 = 0; i0 <= w; i0 += 4) {
            const int i = i0 + sub;
            float d1 = 0.f, d2 = 0.f;
            if (i < w) {
                float kv[per];
                load8(kr + (((size_t)kh * L + i) * KD + part * per) * sa, bf, kv);
                load8(kr + (((size_t)kh * L + i) * KD + part * per + 8) * sa, bf, kv + 8);
#pragma unroll
                for (int u = 0; u < per; ++u) {
                    d1 = fmaf(kv[u], ktv[u], d1);
                    d2 = fmaf(kv[u], qtv[u], d2);
                }
            } else if (i == w) {
#pragma unroll
                for (int u = 0; u < per; ++u) d2 = fmaf(ktv[u], qtv[u], d2);
            }
#pragma unroll
            for (int o = 4; o >= 1; o >>= 1) {
                d1 += __shfl_xor_sync(0xffffffffu, d1, o);
                d2 += __shfl_xor_sync(0xffffffffu, d2, o);
            }
            if (part == 0) {
                if (i < w) {
                    kk[kh * L + i] = d1;
                    kq[kh * L + i] = d2;
                } else if (i == w) {
                    kqt[kh] = d2;
                }
            }
        }
    }
    __syncthreads();

    if (L <= 32) {
        int LS = 1;
        while (LS < L) LS <<= 1;
        const int hpw = 32 / LS;
        const int i = lane & (LS - 1);
        for (int h0 = warp * hpw; h0 < HV; h0 += nwarps * hpw) {
            const int hv = h0 + lane / LS;
            const bool live = hv < HV;
            const float gi = (live && i < w) ? gr[hv * L + i] : 1.f;
            float incl = gi;  // prod_{i<=j<w} g_j after the scan
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                if (off < LS) {
                    const float v = __shfl_down_sync(0xffffffffu, incl, off, LS);
                    if (i + off < LS) incl *= v;
                }
            }
            float gam = __shfl_down_sync(0xffffffffu, incl, 1, LS);  // prod_{i<j<w} g_j
            if (i + 1 >= LS) gam = 1.f;
            const float Gu = __shfl_sync(0xffffffffu, incl, 0, LS);
            if (live) {
                const int kh = hv / vpk;
                const float g_t = gt[hv];
                float* t = a.ws + ((size_t)b * HV + hv) * TBL;
                if (i < L) {
                    const bool hist = i < w;
                    const float Gi = g_t * gam;
                    t[i] = hist ? gam * kk[kh * L + i] : 0.f;
                    t[L + i] = hist ? Gi * kq[kh * L + i] : 0.f;
                    t[2 * L + i] = hist ? Gi : (i == w ? 1.f : 0.f);
                }
                for (int e = 3 * L + i; e < TBL; e += LS) {
                    const int r = e - 3 * L;
                    t[e] = r == 0 ? Gu : r == 1 ? g_t * Gu : r == 2 ? kqt[kh] : r == 3 ? bt[hv]
                         : r == 4 ? g_t : 0.f;
                }
            }
        }
    } else {
        for (int hv = threadIdx.x; hv < HV; hv += blockDim.x) {
            const int kh = hv / vpk;
            const float g_t = gt[hv];
            float* t = a.ws + ((size_t)b * HV + hv) * TBL;
            float gam = 1.f;  // prod_{j=i+1..w-1} g_j
            for (int i = w - 1; i >= 0; --i) {
                const float Gi = g_t * gam;
                t[i] = gam * kk[kh * L + i];
                t[L + i] = Gi * kq[kh * L + i];
                t[2 * L + i] = Gi;
                gam *= gr[hv * L + i];
            }
            for (int i = w; i < L; ++i) {
                t[i] = 0.f;
                t[L + i] = 0.f;
                t[2 * L + i] = (i == w) ? 1.f : 0.f;
            }
            t[3 * L] = gam;
            t[3 * L + 1] = g_t * gam;
            t[3 * L + 2] = kqt[kh];
            t[3 * L + 3] = bt[hv];
            t[3 * L + 4] = g_t;
            for (int i = 3 * L + 5; i < TBL; ++i) t[i] = 0.f;
        }
    }
}

// ----------------------------------------------------------------------------
// prologue kernels
// ----------------------------------------------------------------------------

__global__ void __launch_bounds__(128) ring_append_kernel(const RowArgs a, const int32_t* ci,
                                                          const int32_t* row_wp, int32_t* dev_err) {
    const int b = blockIdx.x;
    const int w = given_cursor(b, ci[b], a.num_slots, a.L, row_wp, threadIdx.x == 0 ? dev_err : nullptr);
    if (w < 0) return;
    append_row(a, b, ci[b], w);
}

__global__ void __launch_bounds__(kRowThreads) precompute_kernel(const RowArgs a, const int32_t* ci,
                                                                 const int32_t* row_wp,
                                                                 int32_t* dev_err) {
    extern __shared__ __align__(128) uint8_t psm[];
    __shared__ uint64_t bar;
    const int b = blockIdx.x;
    const int s = ci[b];
    // bad slots and cursors are reported by the append and output kernels
    const int w = given_cursor(b, s, a.num_slots, a.L, row_wp, nullptr);
    if (w < 0) return;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        stage_issue(a, b, s, psm, &bar);
    }
    __syncthreads();
    if (!mbar_wait_bounded(&bar, 0)) {
        if (threadIdx.x == 0) set_dev_err(dev_err, RSSM_DEVERR_TIMEOUT);
        return;
    }
    tables_from_smem(a, b, w, psm);
}

// Cursor advance (when `advance`), ring append and tables of one row in one CTA.
// Thread 0 issues the staging copies before it reads the cursor. The tables read
// only ring entries before w, so the append needs no ordering with them.
__global__ void __launch_bounds__(kRowThreads) prepare_kernel(const RowArgs a, const int32_t* ci,
                                                              int advance, const uint8_t* force,
                                                              int32_t* slot_wp, int32_t* row_wp,
                                                              uint8_t* row_flush, int32_t* dev_err) {
    extern __shared__ __align__(128) uint8_t psm[];
    __shared__ uint64_t bar;
    __shared__ int sh_w;
    const int b = blockIdx.x;
    const int s = ci[b];
    const bool staged = s >= 0 && s < a.num_slots;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        if (staged) stage_issue(a, b, s, psm, &bar);
        sh_w = advance ? standard_cursor(b, s, a.num_slots, a.L, slot_wp, force, row_wp, row_flush,
                                         dev_err)
                       : given_cursor(b, s, a.num_slots, a.L, row_wp, dev_err);
    }
    __syncthreads();
    const int w = sh_w;
    if (staged && !mbar_wait_bounded(&bar, 0)) {
        if (threadIdx.x == 0) set_dev_err(dev_err, RSSM_DEVERR_TIMEOUT);
        return;
    }
    if (w < 0) return;
    append_row(a, b, s, w);
    tables_from_smem(a, b, w, psm);
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
static int gdn_prologue_smem(const rssm_gdn_dims* d, const void* kernel, int* smem) {
    *smem = gdn::ProLayout(d->num_v_heads, d->num_k_heads, d->ring_len,
                           d->act_dtype == RSSM_BF16 ? 2 : 4).total;
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
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(beta) || !ok_ptr(g) || !ok_ptr(ring_k) ||
        !ok_ptr(ring_g) || !ok_ptr(cache_indices) || !ok_ptr(row_wp) || !ok_ptr(workspace))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_gdn_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    int smem = 0;
    rc = gdn_prologue_smem(d, reinterpret_cast<const void*>(gdn::precompute_kernel), &smem);
    if (rc) return rc;
    gdn::RowArgs ra = gdn::row_args(d);
    ra.q = q;
    ra.k = k;
    ra.beta = beta;
    ra.g = g;
    ra.ring_k = const_cast<void*>(ring_k);  // read only here
    ra.ring_g = const_cast<float*>(ring_g);
    ra.ws = static_cast<float*>(workspace);
    gdn::precompute_kernel<<<d->batch, gdn::kRowThreads, smem, (cudaStream_t)stream>>>(ra, cache_indices,
                                                                                       row_wp, dev_err);
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
    rc = gdn_prologue_smem(d, reinterpret_cast<const void*>(gdn::prepare_kernel), &smem);
    if (rc) return rc;
    gdn::prepare_kernel<<<d->batch, gdn::kRowThreads, smem, (cudaStream_t)stream>>>(
        ra, cache_indices, adv, force_flush, slot_wp, row_wp, row_flush, dev_err);
    return launch_status();
}
