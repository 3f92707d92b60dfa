// gdn.cu -- ReplaySSM decode for the gated delta net on sm_103a.
//
// Pages followed: [GDN] "GDN ReplaySSM decode (Part A of RFC 28511)" (SGLang PR
// 28451 report): 功能与动机 (the conventional decode kernel reads and writes the
// full state [HV, V, K] every step and is bandwidth bound at batch >= 64;
// ReplaySSM removes the per-step state write), 实现拆解 item 1 (the decode kernel
// reconstructs non-flush outputs from the checkpoint S0 plus the (d, k, g) ring
// and flushes the full state every L steps), 实现拆解 item 3 (the ring tensors
// d, k, g per slot). [SPEC] "[GDN] Support ReplaySSM Ring Spec-Verify",
// 风险与影响: the checkpoint is fp32.
//
// Recurrence per value head (key head kh = hv / (HV/HK)):
//   S <- g S + beta (v - g S k) k^T,  o = S q.
// Unrolled from the checkpoint S0 over ring entries i < w and the current step:
//   u   = S_{t-1} k_t = Gu (S0 k_t) + sum_{i<w} gamma_i (k_i . k_t) d_i
//   d_t = beta_t (v_t - g_t u)
//   o   = Go (S0 q_t) + sum_{i<w} Gamma_i (k_i . q_t) d_i + (k_t . q_t) d_t
//   flush: S = Go S0 + sum_{i<=w} Gamma_i d_i k_i^T
// with gamma_i = prod_{j=i+1..w-1} g_j, Gamma_i = g_t gamma_i (Gamma_w = 1),
// Gu = prod_{j<w} g_j, Go = g_t Gu.
//
// Work item of the output kernel = (row, value head, block of 32 value rows): a
// 16 KB fp32 tile of S0, read by a group of two consumer warps. Each warp owns 16
// value rows; a lane holds 4 key columns of a row (16-byte shared loads), so the
// two dot products per row reduce across the warp with one 32-way reduce-scatter.
// The d ring is stored in blocks of 32 value rows, so a block's history entries
// arrive with one bulk copy. The per-row prologue kernels (ring append, tables)
// are in gdn_prologue.cu.
#include "common.cuh"
#include "gdn.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace rssm {
namespace gdn {

// ----------------------------------------------------------------------------
// output / flush and full-state decode (warp-specialised pipeline)
// ----------------------------------------------------------------------------
//
// A group of two consumer warps owns a (row, value head, 32-row block) tile, 16
// value rows per warp; lane l holds key columns 4l..4l+3 of every row, so one
// 16-byte shared load per lane reads one value row. The two dot products per row
// (with k_t and q_t) of 16 rows reduce with one 32-way reduce-scatter; lanes 0..15
// then own rows base + lane.

constexpr int kGroupWarps = 2;
constexpr int RW = VB / kGroupWarps;  // value rows per warp

struct OutPolicy {
    static constexpr int kGroup = kGroupWarps;
    struct Args {
        float* state;
        const void* q;
        const void* v;
        const void* ring_k;
        float* ring_d;
        const int32_t* ci;
        const int32_t* row_wp;
        const uint8_t* row_flush;
        const float* ws;
        void* o;
        int32_t* dev_err;
        int batch, HV, HK, V, L, num_slots, act_bf16, out_bf16;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
        int off_k, off_q, off_v, off_d, off_tbl;
    };
    struct Meta {
        int valid, s, b, hv, vb, w, f;
    };

    static __device__ int n_items(const Args& a) { return a.batch * a.HV * (a.V / VB); }

    static __device__ int4 prefetch(const Args& a, int item) {
        const int b = item / (a.HV * (a.V / VB));
        const int s = a.ci[b];
        int w = 0, f = 0;
        if (s >= 0 && s < a.num_slots) {
            w = a.row_wp[b];
            f = a.row_flush[b];
        }
        return make_int4(s, w, f, b);
    }

    static __device__ void issue(const Args& a, int item, int4 r, Meta* meta, uint8_t* sb,
                                 uint64_t* full, uint64_t pol) {
        const int NVB = a.V / VB;
        const int b = r.w;
        const int rem = item - b * a.HV * NVB;
        const int hv = rem / NVB, vb = rem - (rem / NVB) * NVB;
        Meta m{0, r.x, b, hv, vb, r.y, r.z};
        if (r.x >= a.num_slots) {
            set_dev_err(a.dev_err, RSSM_DEVERR_SLOT);
        } else if (r.x >= 0) {
            if (r.y < 0 || r.y >= a.L) set_dev_err(a.dev_err, RSSM_DEVERR_CURSOR);
            else m.valid = 1;
        }
        *meta = m;
        if (!m.valid) {
            mbar_arrive_plain(full);
            return;
        }
        const int sa = a.act_bf16 ? 2 : 4;
        const int L = a.L, w = m.w;
        const int kh = hv / (a.HV / a.HK);
        const int TBL = tbl_floats(L);
        const uint32_t kb = KD * sa;
        const uint32_t kbytes = m.f ? (w + 1) * kb : kb;
        mbar_arrive_expect_tx(full, TILE + kbytes + kb + VB * sa + w * VB * 4 + TBL * 4);
        bulk_g2s_hint(sb, a.state + (((size_t)m.s * a.HV + hv) * a.V + (size_t)vb * VB) * KD, TILE,
                      full, pol);
        const char* kr = static_cast<const char*>(a.ring_k) + ((size_t)m.s * a.HK + kh) * L * kb;
        if (m.f) bulk_g2s(sb + a.off_k, kr, kbytes, full);
        else bulk_g2s(sb + a.off_k + w * kb, kr + (size_t)w * kb, kb, full);
        bulk_g2s(sb + a.off_q, static_cast<const char*>(a.q) + ((size_t)b * a.HK + kh) * kb, kb, full);
        bulk_g2s(sb + a.off_v,
                 static_cast<const char*>(a.v) + (((size_t)b * a.HV + hv) * a.V + (size_t)vb * VB) * sa,
                 VB * sa, full);
        // ring d is blocked by 32 value rows: the block's entries 0..w-1 are contiguous
        if (w > 0)
            bulk_g2s(sb + a.off_d, a.ring_d + ((((size_t)m.s * a.HV + hv) * NVB + vb) * L) * VB,
                     w * VB * 4, full);
        bulk_g2s(sb + a.off_tbl, a.ws + ((size_t)b * a.HV + hv) * TBL, TBL * 4, full);
    }

    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb, uint8_t*,
                                   int lane, int wi) {
        if (!m.valid) return;
        const bool bf = a.act_bf16;
        const int sa = bf ? 2 : 4;
        const int L = a.L, w = m.w;
        const int rbase = wi * RW;
        const float* tile = reinterpret_cast<const float*>(sb);
        const uint8_t* kring = sb + a.off_k;
        const float* dring = reinterpret_cast<const float*>(sb + a.off_d);
        const float* t = reinterpret_cast<const float*>(sb + a.off_tbl);
        float k4[4], q4[4];
        load4(kring + (size_t)w * KD * sa, lane * 4, bf, k4);
        load4(sb + a.off_q, lane * 4, bf, q4);
        constexpr int NCHK = RW / 16;
        float av[NCHK], cv[NCHK];
#pragma unroll
        for (int ch = 0; ch < NCHK; ++ch) {
            float part[32];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float4 s4 =
                    *reinterpret_cast<const float4*>(tile + (rbase + ch * 16 + j) * KD + lane * 4);
                part[j] = s4.x * k4[0] + s4.y * k4[1] + s4.z * k4[2] + s4.w * k4[3];
                part[16 + j] = s4.x * q4[0] + s4.y * q4[1] + s4.z * q4[2] + s4.w * q4[3];
            }
            reduce_scatter<32, 32>(part);  // lane l holds entry l
            av[ch] = part[0];
            cv[ch] = __shfl_down_sync(kFull, part[0], 16);
        }
        const float Gu = t[3 * L], Go = t[3 * L + 1], kqt = t[3 * L + 2];
        const float bt = t[3 * L + 3], gt = t[3 * L + 4];
        float dtv[NCHK];
#pragma unroll
        for (int ch = 0; ch < NCHK; ++ch) {
            dtv[ch] = 0.f;
            if (lane < 16) {
                const int r = rbase + ch * 16 + lane;
                float u = Gu * av[ch];
                float oo = Go * cv[ch];
                for (int i = 0; i < w; ++i) {
                    const float di = dring[i * VB + r];
                    u = fmaf(t[i], di, u);
                    oo = fmaf(t[L + i], di, oo);
                }
                const float dn = bt * (load1(sb + a.off_v, r, bf) - gt * u);
                oo = fmaf(kqt, dn, oo);
                const size_t vi = (size_t)m.vb * VB + r;
                store1(a.o, ((size_t)m.b * a.HV + m.hv) * a.V + vi, a.out_bf16, oo);
                a.ring_d[((((size_t)m.s * a.HV + m.hv) * (a.V / VB) + m.vb) * L + w) * VB + r] = dn;
                dtv[ch] = dn;
            }
        }
        if (m.f) {
            // S = Go S0 + sum_{i<=w} Gamma_i d_i k_i^T (d_w = this step's d)
            float* dst = a.state + (((size_t)m.s * a.HV + m.hv) * a.V + (size_t)m.vb * VB) * KD;
#pragma unroll 1
            for (int hb = 0; hb < 2 * NCHK; ++hb) {  // blocks of 8 value rows
                const int r0 = rbase + hb * 8;
                const float dsrc = (hb >> 1) == 0 ? dtv[0] : dtv[NCHK - 1];
                float dcur[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) dcur[j] = __shfl_sync(kFull, dsrc, (hb & 1) * 8 + j);
                float acc[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 s4 = *reinterpret_cast<const float4*>(tile + (r0 + j) * KD + lane * 4);
                    acc[j][0] = Go * s4.x; acc[j][1] = Go * s4.y;
                    acc[j][2] = Go * s4.z; acc[j][3] = Go * s4.w;
                }
                for (int i = 0; i <= w; ++i) {
                    float ki[4];
                    load4(kring + (size_t)i * KD * sa, lane * 4, bf, ki);
                    const float ti = t[2 * L + i];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float dj = (i < w) ? dring[i * VB + r0 + j] : dcur[j];
                        const float c = ti * dj;
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[j][e] = fmaf(c, ki[e], acc[j][e]);
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4*>(dst + (r0 + j) * KD + lane * 4) =
                        make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
            }
        }
    }
};

struct FullPolicy {
    static constexpr int kGroup = kGroupWarps;
    struct Args {
        float* state;
        const void* q;
        const void* k;
        const void* v;
        const float* beta;
        const float* g;
        const int32_t* ci;
        void* o;
        int32_t* dev_err;
        int batch, HV, HK, V, num_slots, act_bf16, out_bf16;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
        int off_k, off_q, off_v;
    };
    struct Meta {
        int valid, s, b, hv, vb;
        float beta, g;
    };

    static __device__ int n_items(const Args& a) { return a.batch * a.HV * (a.V / VB); }

    static __device__ int4 prefetch(const Args& a, int item) {
        const int NVB = a.V / VB;
        const int b = item / (a.HV * NVB);
        const int hv = (item - b * a.HV * NVB) / NVB;
        const int s = a.ci[b];
        float be = 0.f, gg = 0.f;
        if (s >= 0 && s < a.num_slots) {
            be = a.beta[(size_t)b * a.HV + hv];
            gg = a.g[(size_t)b * a.HV + hv];
        }
        return make_int4(s, b, __float_as_int(be), __float_as_int(gg));
    }

    static __device__ void issue(const Args& a, int item, int4 r, Meta* meta, uint8_t* sb,
                                 uint64_t* full, uint64_t pol) {
        const int NVB = a.V / VB;
        const int b = r.y;
        const int rem = item - b * a.HV * NVB;
        const int hv = rem / NVB, vb = rem - (rem / NVB) * NVB;
        Meta m{0, r.x, b, hv, vb, __int_as_float(r.z), __int_as_float(r.w)};
        if (r.x >= a.num_slots) set_dev_err(a.dev_err, RSSM_DEVERR_SLOT);
        else if (r.x >= 0) m.valid = 1;
        *meta = m;
        if (!m.valid) {
            mbar_arrive_plain(full);
            return;
        }
        const int sa = a.act_bf16 ? 2 : 4;
        const int kh = hv / (a.HV / a.HK);
        const uint32_t kb = KD * sa;
        mbar_arrive_expect_tx(full, TILE + 2 * kb + VB * sa);
        bulk_g2s_hint(sb, a.state + (((size_t)m.s * a.HV + hv) * a.V + (size_t)vb * VB) * KD, TILE,
                      full, pol);
        bulk_g2s(sb + a.off_k, static_cast<const char*>(a.k) + ((size_t)b * a.HK + kh) * kb, kb, full);
        bulk_g2s(sb + a.off_q, static_cast<const char*>(a.q) + ((size_t)b * a.HK + kh) * kb, kb, full);
        bulk_g2s(sb + a.off_v,
                 static_cast<const char*>(a.v) + (((size_t)b * a.HV + hv) * a.V + (size_t)vb * VB) * sa,
                 VB * sa, full);
    }

    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb, uint8_t*,
                                   int lane, int wi) {
        if (!m.valid) return;
        const bool bf = a.act_bf16;
        const float* tile = reinterpret_cast<const float*>(sb);
        float k4[4], q4[4];
        load4(sb + a.off_k, lane * 4, bf, k4);
        load4(sb + a.off_q, lane * 4, bf, q4);
        float kq = k4[0] * q4[0] + k4[1] * q4[1] + k4[2] * q4[2] + k4[3] * q4[3];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) kq += __shfl_xor_sync(kFull, kq, o);
        float* dst = a.state + (((size_t)m.s * a.HV + m.hv) * a.V + (size_t)m.vb * VB) * KD;
#pragma unroll 1
        for (int ch = 0; ch < RW / 16; ++ch) {
            const int r0 = wi * RW + ch * 16;
            float part[32];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float4 s4 = *reinterpret_cast<const float4*>(tile + (r0 + j) * KD + lane * 4);
                part[j] = s4.x * k4[0] + s4.y * k4[1] + s4.z * k4[2] + s4.w * k4[3];
                part[16 + j] = s4.x * q4[0] + s4.y * q4[1] + s4.z * q4[2] + s4.w * q4[3];
            }
            reduce_scatter<32, 32>(part);
            const float cdot = __shfl_down_sync(kFull, part[0], 16);
            float dn = 0.f;
            if (lane < 16) {
                const int r = r0 + lane;
                dn = m.beta * (load1(sb + a.off_v, r, bf) - m.g * part[0]);
                const float oo = m.g * cdot + dn * kq;
                store1(a.o, ((size_t)m.b * a.HV + m.hv) * a.V + (size_t)m.vb * VB + r, a.out_bf16, oo);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float dj = __shfl_sync(kFull, dn, j);
                float4 s4 = *reinterpret_cast<const float4*>(tile + (r0 + j) * KD + lane * 4);
                s4.x = fmaf(m.g, s4.x, dj * k4[0]);
                s4.y = fmaf(m.g, s4.y, dj * k4[1]);
                s4.z = fmaf(m.g, s4.z, dj * k4[2]);
                s4.w = fmaf(m.g, s4.w, dj * k4[3]);
                *reinterpret_cast<float4*>(dst + (r0 + j) * KD + lane * 4) = s4;
            }
        }
    }
};

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------

int check_dims(const rssm_gdn_dims* d) {
    if (!d) return RSSM_ERR_INVALID_ARG;
    if (d->batch < 0 || d->num_v_heads <= 0 || d->num_k_heads <= 0 || d->head_k_dim <= 0 ||
        d->head_v_dim <= 0 || d->num_slots <= 0)
        return RSSM_ERR_INVALID_ARG;
    if (!ok_dtype(d->act_dtype) || !ok_dtype(d->out_dtype)) return RSSM_ERR_INVALID_ARG;
    if (d->ring_len < 1 || d->num_v_heads % d->num_k_heads) return RSSM_ERR_CONFIG;
    if (d->head_k_dim != KD || d->head_v_dim % VB) return RSSM_ERR_UNSUPPORTED;
    return RSSM_OK;
}

}  // namespace gdn
}  // namespace rssm

using namespace rssm;

extern "C" int rssm_gdn_output(const rssm_gdn_dims* d, float* state, const void* q, const void* v,
                               const void* ring_k, float* ring_d, const int32_t* cache_indices,
                               const int32_t* row_wp, const uint8_t* row_flush,
                               const void* workspace, size_t workspace_bytes, void* o,
                               int32_t* dev_err, rssm_stream_t stream) {
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(q) || !ok_ptr(v) || !ok_ptr(ring_k) || !ok_ptr(ring_d) ||
        !ok_ptr(cache_indices) || !ok_ptr(row_wp) || !ok_ptr(row_flush) || !ok_ptr(workspace) ||
        !ok_ptr(o))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_gdn_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    gdn::OutPolicy::Args a{};
    a.state = state; a.q = q; a.v = v; a.ring_k = ring_k; a.ring_d = ring_d; a.ci = cache_indices;
    a.row_wp = row_wp; a.row_flush = row_flush; a.ws = static_cast<const float*>(workspace);
    a.o = o; a.dev_err = dev_err;
    a.batch = d->batch; a.HV = d->num_v_heads; a.HK = d->num_k_heads; a.V = d->head_v_dim;
    a.L = d->ring_len; a.num_slots = d->num_slots; a.act_bf16 = d->act_dtype == RSSM_BF16;
    a.out_bf16 = d->out_dtype == RSSM_BF16;
    const int sa = a.act_bf16 ? 2 : 4;
    int off = gdn::TILE;
    a.off_k = off;   off += a.L * gdn::KD * sa;
    a.off_q = off;   off += gdn::KD * sa;
    a.off_v = off;   off += gdn::VB * sa;
    a.off_d = off;   off += a.L * gdn::VB * 4;
    a.off_tbl = off; off += gdn::tbl_floats(a.L) * 4;
    const int stage_bytes = (off + 127) & ~127;
    return launch_pipe<gdn::OutPolicy>(a, stage_bytes, 0, gdn::TILE,
                                       (long)d->batch * d->num_v_heads * (d->head_v_dim / gdn::VB),
                                       (cudaStream_t)stream);
}

extern "C" int rssm_gdn_decode(const rssm_gdn_dims* d, float* state, const void* q, const void* k,
                               const void* v, const float* beta, const float* g,
                               const void* ring_k, const float* ring_g, float* ring_d,
                               const int32_t* cache_indices, const int32_t* row_wp,
                               const uint8_t* row_flush, void* workspace, size_t workspace_bytes,
                               void* o, int32_t* dev_err, rssm_stream_t stream) {
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(beta) || !ok_ptr(g) ||
        !ok_ptr(ring_k) || !ok_ptr(ring_g) || !ok_ptr(ring_d) || !ok_ptr(cache_indices) ||
        !ok_ptr(row_wp) || !ok_ptr(row_flush) || !ok_ptr(workspace) || !ok_ptr(o))
        return RSSM_ERR_INVALID_ARG;
    rc = rssm_gdn_precompute(d, q, k, beta, g, ring_k, ring_g, cache_indices, row_wp, workspace,
                             workspace_bytes, dev_err, stream);
    if (rc) return rc;
    return rssm_gdn_output(d, state, q, v, ring_k, ring_d, cache_indices, row_wp, row_flush,
                           workspace, workspace_bytes, o, dev_err, stream);
}

extern "C" int rssm_gdn_step(const rssm_gdn_dims* d, int advance, const uint8_t* force_flush,
                             int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush, float* state,
                             const void* q, const void* k, const void* v, const float* beta,
                             const float* g, const int32_t* cache_indices, void* ring_k,
                             float* ring_g, float* ring_d, void* workspace,
                             size_t workspace_bytes, void* o, int32_t* dev_err,
                             rssm_stream_t stream) {
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(v) || !ok_ptr(ring_d) || !ok_ptr(o) || !ok_ptr(row_flush))
        return RSSM_ERR_INVALID_ARG;
    rc = rssm_gdn_prepare(d, advance, force_flush, slot_wp, row_wp, row_flush, q, k, beta, g,
                          cache_indices, ring_k, ring_g, workspace, workspace_bytes, dev_err,
                          stream);
    if (rc) return rc;
    return rssm_gdn_output(d, state, q, v, ring_k, ring_d, cache_indices, row_wp, row_flush,
                           workspace, workspace_bytes, o, dev_err, stream);
}

extern "C" int rssm_gdn_full_state_decode(const rssm_gdn_dims* d, float* state, const void* q,
                                          const void* k, const void* v, const float* beta,
                                          const float* g, const int32_t* cache_indices, void* o,
                                          int32_t* dev_err, rssm_stream_t stream) {
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(beta) || !ok_ptr(g) ||
        !ok_ptr(cache_indices) || !ok_ptr(o))
        return RSSM_ERR_INVALID_ARG;
    gdn::FullPolicy::Args a{};
    a.state = state; a.q = q; a.k = k; a.v = v; a.beta = beta; a.g = g; a.ci = cache_indices;
    a.o = o; a.dev_err = dev_err;
    a.batch = d->batch; a.HV = d->num_v_heads; a.HK = d->num_k_heads; a.V = d->head_v_dim;
    a.num_slots = d->num_slots; a.act_bf16 = d->act_dtype == RSSM_BF16;
    a.out_bf16 = d->out_dtype == RSSM_BF16;
    const int sa = a.act_bf16 ? 2 : 4;
    int off = gdn::TILE;
    a.off_k = off; off += gdn::KD * sa;
    a.off_q = off; off += gdn::KD * sa;
    a.off_v = off; off += gdn::VB * sa;
    const int stage_bytes = (off + 127) & ~127;
    return launch_pipe<gdn::FullPolicy>(a, stage_bytes, 0, gdn::TILE,
                                        (long)d->batch * d->num_v_heads * (d->head_v_dim / gdn::VB),
                                        (cudaStream_t)stream);
}
