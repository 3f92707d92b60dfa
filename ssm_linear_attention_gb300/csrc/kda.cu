// kda.cu -- ReplaySSM decode for the gated delta rule with a per-key-channel gate
// (KDA) on sm_103a.
//
// Pages followed: "GDN ReplaySSM decode (Part A of RFC 28511)" (SGLang PR 28451
// report): 实现拆解 item 1 (one buffered decode kernel serves the scalar GDN gate
// and the KDA per-K gate, IS_KDA) and 评论区精华 (the KDA gate ring g_cache
// [slots, HV, L, K] makes each step's ring write larger; the report measured no
// gain for KDA and left the reason open).
//
// Recurrence per value head (key head kh = hv / (HV/HK)), a_t in (0, 1]^K:
//   S <- S Diag(a_t) + beta_t (v_t - S Diag(a_t) k_t) k_t^T,  o = S q_t.
// With Gam_m = prod_{j=m+1..w} a_j (per channel; Gam_w = 1) and Gam_{-1} =
// prod_{j=0..w} a_j, unrolling from the checkpoint S0 over ring entries m < w and
// the current step w gives
//   u   = S0 (Gam_{-1} o k_w) + sum_{m<w} kk_m d_m,   kk_m = k_m . (Gam_m o k_w)
//   d_w = beta_w (v_w - u)
//   o   = S0 (Gam_{-1} o q_w) + sum_{m<=w} kq_m d_m,  kq_m = k_m . (Gam_m o q_w)
//   flush: S = S0 Diag(Gam_{-1}) + sum_{m<=w} d_m (Gam_m o k_m)^T
// (o = element-wise product). The prologue builds, per (row, value head), the two
// gated vectors, Gam_{-1}, the kk / kq tables and, on flush rows, the gated keys;
// the output kernel streams the checkpoint tile once and needs nothing per
// channel beyond two 512-byte vectors.
#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace rssm {
namespace kda {

constexpr int KD = 128;  // key dim
constexpr int VB = 32;   // value rows per output work item
constexpr int TILE = VB * KD * 4;
constexpr int kGroupWarps = 2;
constexpr int RW = VB / kGroupWarps;
constexpr int kMaxL = 64;

// Workspace: [batch][HV][main_floats(L)] then [batch][HV][L][KD] (gated keys of
// flush rows). main = ku[KD], qo[KD], gam[KD], kk[L], kq[L], beta, padded to 4.
__host__ __device__ inline int main_floats(int L) { return 3 * KD + ((2 * L + 1 + 3) & ~3); }

inline size_t kg_offset_floats(const rssm_gdn_dims* d) {
    return (size_t)d->batch * d->num_v_heads * main_floats(d->ring_len);
}

int check_dims(const rssm_gdn_dims* d) {
    if (!d) return RSSM_ERR_INVALID_ARG;
    if (d->batch < 0 || d->num_v_heads <= 0 || d->num_k_heads <= 0 || d->head_k_dim <= 0 ||
        d->head_v_dim <= 0 || d->num_slots <= 0)
        return RSSM_ERR_INVALID_ARG;
    if (!ok_dtype(d->act_dtype) || !ok_dtype(d->out_dtype)) return RSSM_ERR_INVALID_ARG;
    if (d->ring_len < 1 || d->num_v_heads % d->num_k_heads) return RSSM_ERR_CONFIG;
    if (d->head_k_dim != KD || d->head_v_dim % VB || d->ring_len > kMaxL) return RSSM_ERR_UNSUPPORTED;
    return RSSM_OK;
}

// ----------------------------------------------------------------------------
// prologue: ring append and tables, one warp per (row, value head)
// ----------------------------------------------------------------------------

constexpr int kPreWarps = 4;  // (row, value head) items per CTA
constexpr int kChunkM = 16;   // ring entries whose dot products reduce together

struct PreArgs {
    const void* q;
    const void* k;
    const float* a;
    const float* beta;
    const int32_t* ci;
    const int32_t* row_wp;
    const uint8_t* row_flush;
    void* ring_k;
    float* ring_a;
    float* ws;
    float* ws_kg;
    int32_t* dev_err;
    int n_items, HV, HK, L, num_slots, act_bf16;
};

// Lane l owns key channels 4l..4l+3. The ring entries are visited from the current
// one (m = w) down to 0, carrying Gam_m per channel; the partial dot products of up
// to 16 entries reduce together with one 32-way reduce-scatter (lanes 0..15 end up
// with k_m . (Gam_m o k_t), lanes 16..31 with k_m . (Gam_m o q_t)).
__global__ void __launch_bounds__(32 * kPreWarps) prepare_kernel(const PreArgs a) {
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * kPreWarps + (threadIdx.x >> 5);
    if (item >= a.n_items) return;
    const int L = a.L;
    const int b = item / a.HV, hv = item - (item / a.HV) * a.HV;
    const int vpk = a.HV / a.HK, kh = hv / vpk;
    const int s = a.ci[b];
    if (s < 0) return;
    if (s >= a.num_slots) {
        if (lane == 0 && hv == 0) set_dev_err(a.dev_err, RSSM_DEVERR_SLOT);
        return;
    }
    const int w = a.row_wp[b];
    if (w < 0 || w >= L) {
        if (lane == 0 && hv == 0) set_dev_err(a.dev_err, RSSM_DEVERR_CURSOR);
        return;
    }
    const int f = a.row_flush[b];
    const bool bf = a.act_bf16;
    const int c4 = lane * 4;
    const float* ra = a.ring_a + ((size_t)s * a.HV + hv) * L * KD;
    const size_t rk = ((size_t)s * a.HK + kh) * L * KD;
    const float4 aw = *reinterpret_cast<const float4*>(a.a + ((size_t)b * a.HV + hv) * KD + c4);
    const int sa = bf ? 2 : 4;
    const char* krow = static_cast<const char*>(a.ring_k) + rk * sa;  // this key head's ring
    float kw[4], qw[4];
    load4(static_cast<const char*>(a.k) + ((size_t)b * a.HK + kh) * KD * sa, c4, bf, kw);
    load4(static_cast<const char*>(a.q) + ((size_t)b * a.HK + kh) * KD * sa, c4, bf, qw);
    // ring append (the k entry once per key head)
    *reinterpret_cast<float4*>(a.ring_a + ((size_t)s * a.HV + hv) * L * KD + (size_t)w * KD + c4) = aw;
    if (hv % vpk == 0) {
        char* kd = static_cast<char*>(a.ring_k) + (rk + (size_t)w * KD + c4) * sa;
        if (bf) {
            *reinterpret_cast<uint2*>(kd) =
                make_uint2(pack_bf16x2(kw[0], kw[1]), pack_bf16x2(kw[2], kw[3]));
        } else {
            *reinterpret_cast<float4*>(kd) = make_float4(kw[0], kw[1], kw[2], kw[3]);
        }
    }

    float* wsm = a.ws + ((size_t)b * a.HV + hv) * main_floats(L);
    float* tb = wsm + 3 * KD;
    float* kgo = a.ws_kg + ((size_t)b * a.HV + hv) * L * KD;
    float G[4] = {1.f, 1.f, 1.f, 1.f};  // Gam_m of the entry being visited
    // chunks of entries [m0, m0 + 16) from the top: m0 = 16 * floor(w / 16), ..., 0
    for (int m0 = (w / kChunkM) * kChunkM; m0 >= 0; m0 -= kChunkM) {
        float part[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) part[j] = 0.f;
#pragma unroll
        for (int jj = kChunkM - 1; jj >= 0; --jj) {
            const int m = m0 + jj;
            if (m <= w) {
                float km[4], am[4];
                if (m == w) {
                    km[0] = kw[0]; km[1] = kw[1]; km[2] = kw[2]; km[3] = kw[3];
                    am[0] = aw.x; am[1] = aw.y; am[2] = aw.z; am[3] = aw.w;
                } else {
                    load4(krow + (size_t)m * KD * sa, c4, bf, km);
                    const float4 a4 = *reinterpret_cast<const float4*>(ra + (size_t)m * KD + c4);
                    am[0] = a4.x; am[1] = a4.y; am[2] = a4.z; am[3] = a4.w;
                }
                float gk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) gk[e] = G[e] * km[e];
                if (f)
                    *reinterpret_cast<float4*>(kgo + (size_t)m * KD + c4) =
                        make_float4(gk[0], gk[1], gk[2], gk[3]);
                part[jj] = gk[0] * kw[0] + gk[1] * kw[1] + gk[2] * kw[2] + gk[3] * kw[3];
                part[16 + jj] = gk[0] * qw[0] + gk[1] * qw[1] + gk[2] * qw[2] + gk[3] * qw[3];
#pragma unroll
                for (int e = 0; e < 4; ++e) G[e] *= am[e];
            }
        }
        reduce_scatter<32, 32>(part);  // lane l holds entry l
        const int m = m0 + (lane & 15);
        if (m <= w) tb[(lane >> 4) * L + m] = part[0];  // kk_m / kq_m
    }
    // G = Gam_{-1}
    *reinterpret_cast<float4*>(wsm + c4) = make_float4(G[0] * kw[0], G[1] * kw[1], G[2] * kw[2], G[3] * kw[3]);
    *reinterpret_cast<float4*>(wsm + KD + c4) =
        make_float4(G[0] * qw[0], G[1] * qw[1], G[2] * qw[2], G[3] * qw[3]);
    *reinterpret_cast<float4*>(wsm + 2 * KD + c4) = make_float4(G[0], G[1], G[2], G[3]);
    if (lane == 0) tb[2 * L] = a.beta[(size_t)b * a.HV + hv];
}

// ----------------------------------------------------------------------------
// output / flush (warp-specialised pipeline; 16 value rows per consumer warp,
// lane l holds key channels 4l..4l+3)
// ----------------------------------------------------------------------------

struct OutPolicy {
    static constexpr int kGroup = kGroupWarps;
    struct Args {
        float* state;
        const void* v;
        float* ring_d;
        const int32_t* ci;
        const int32_t* row_wp;
        const uint8_t* row_flush;
        const float* ws;
        const float* ws_kg;
        void* o;
        int32_t* dev_err;
        int batch, HV, V, L, num_slots, act_bf16, out_bf16;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
        int off_vec, off_v, off_d;
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
        const uint32_t mainb = main_floats(L) * 4;
        mbar_arrive_expect_tx(full, TILE + mainb + VB * sa + w * VB * 4);
        bulk_g2s_hint(sb, a.state + (((size_t)m.s * a.HV + hv) * a.V + (size_t)vb * VB) * KD, TILE,
                      full, pol);
        bulk_g2s(sb + a.off_vec, a.ws + ((size_t)b * a.HV + hv) * main_floats(L), mainb, full);
        bulk_g2s(sb + a.off_v,
                 static_cast<const char*>(a.v) + (((size_t)b * a.HV + hv) * a.V + (size_t)vb * VB) * sa,
                 VB * sa, full);
        if (w > 0)
            bulk_g2s(sb + a.off_d, a.ring_d + ((((size_t)m.s * a.HV + hv) * NVB + vb) * L) * VB,
                     w * VB * 4, full);
    }

    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb, uint8_t*,
                                   int lane, int wi) {
        if (!m.valid) return;
        const bool bf = a.act_bf16;
        const int L = a.L, w = m.w;
        const int rbase = wi * RW;
        const float* tile = reinterpret_cast<const float*>(sb);
        const float* vec = reinterpret_cast<const float*>(sb + a.off_vec);
        const float* tb = vec + 3 * KD;  // kk[L], kq[L], beta
        const float* dring = reinterpret_cast<const float*>(sb + a.off_d);
        const float4 ku = *reinterpret_cast<const float4*>(vec + lane * 4);
        const float4 qo = *reinterpret_cast<const float4*>(vec + KD + lane * 4);
        float part[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float4 s4 = *reinterpret_cast<const float4*>(tile + (rbase + j) * KD + lane * 4);
            part[j] = s4.x * ku.x + s4.y * ku.y + s4.z * ku.z + s4.w * ku.w;
            part[16 + j] = s4.x * qo.x + s4.y * qo.y + s4.z * qo.z + s4.w * qo.w;
        }
        reduce_scatter<32, 32>(part);  // lane l holds entry l
        const float cdot = __shfl_down_sync(kFull, part[0], 16);
        float dn = 0.f;
        if (lane < 16) {
            const int r = rbase + lane;
            float u = part[0], oo = cdot;
            for (int i = 0; i < w; ++i) {
                const float di = dring[i * VB + r];
                u = fmaf(tb[i], di, u);
                oo = fmaf(tb[L + i], di, oo);
            }
            dn = tb[2 * L] * (load1(sb + a.off_v, r, bf) - u);
            oo = fmaf(tb[L + w], dn, oo);
            const size_t vi = (size_t)m.vb * VB + r;
            store1(a.o, ((size_t)m.b * a.HV + m.hv) * a.V + vi, a.out_bf16, oo);
            a.ring_d[((((size_t)m.s * a.HV + m.hv) * (a.V / VB) + m.vb) * L + w) * VB + r] = dn;
        }
        if (m.f) {
            // S = S0 Diag(Gam_{-1}) + sum_{i<=w} d_i (Gam_i o k_i)^T; the gated keys
            // come from the prologue's workspace (L2)
            const float4 gm = *reinterpret_cast<const float4*>(vec + 2 * KD + lane * 4);
            const float* kg = a.ws_kg + ((size_t)m.b * a.HV + m.hv) * L * KD;
            float* dst = a.state + (((size_t)m.s * a.HV + m.hv) * a.V + (size_t)m.vb * VB) * KD;
#pragma unroll 1
            for (int hb = 0; hb < 2; ++hb) {  // blocks of 8 value rows
                const int r0 = rbase + hb * 8;
                float dcur[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) dcur[j] = __shfl_sync(kFull, dn, hb * 8 + j);
                float acc[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 s4 = *reinterpret_cast<const float4*>(tile + (r0 + j) * KD + lane * 4);
                    acc[j][0] = gm.x * s4.x; acc[j][1] = gm.y * s4.y;
                    acc[j][2] = gm.z * s4.z; acc[j][3] = gm.w * s4.w;
                }
                for (int i = 0; i <= w; ++i) {
                    const float4 k4 = *reinterpret_cast<const float4*>(kg + (size_t)i * KD + lane * 4);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float dj = (i < w) ? dring[i * VB + r0 + j] : dcur[j];
                        acc[j][0] = fmaf(dj, k4.x, acc[j][0]);
                        acc[j][1] = fmaf(dj, k4.y, acc[j][1]);
                        acc[j][2] = fmaf(dj, k4.z, acc[j][2]);
                        acc[j][3] = fmaf(dj, k4.w, acc[j][3]);
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

// ----------------------------------------------------------------------------
// the conventional full-state step (comparison)
// ----------------------------------------------------------------------------

struct FullPolicy {
    static constexpr int kGroup = kGroupWarps;
    struct Args {
        float* state;
        const void* q;
        const void* k;
        const void* v;
        const float* beta;
        const float* a;
        const int32_t* ci;
        void* o;
        int32_t* dev_err;
        int batch, HV, HK, V, num_slots, act_bf16, out_bf16;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
        int off_k, off_q, off_v, off_a;
    };
    struct Meta {
        int valid, s, b, hv, vb;
        float beta;
    };

    static __device__ int n_items(const Args& a) { return a.batch * a.HV * (a.V / VB); }

    static __device__ int4 prefetch(const Args& a, int item) {
        const int NVB = a.V / VB;
        const int b = item / (a.HV * NVB);
        const int hv = (item - b * a.HV * NVB) / NVB;
        const int s = a.ci[b];
        float be = 0.f;
        if (s >= 0 && s < a.num_slots) be = a.beta[(size_t)b * a.HV + hv];
        return make_int4(s, b, __float_as_int(be), 0);
    }

    static __device__ void issue(const Args& a, int item, int4 r, Meta* meta, uint8_t* sb,
                                 uint64_t* full, uint64_t pol) {
        const int NVB = a.V / VB;
        const int b = r.y;
        const int rem = item - b * a.HV * NVB;
        const int hv = rem / NVB, vb = rem - (rem / NVB) * NVB;
        Meta m{0, r.x, b, hv, vb, __int_as_float(r.z)};
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
        mbar_arrive_expect_tx(full, TILE + 2 * kb + VB * sa + KD * 4);
        bulk_g2s_hint(sb, a.state + (((size_t)m.s * a.HV + hv) * a.V + (size_t)vb * VB) * KD, TILE,
                      full, pol);
        bulk_g2s(sb + a.off_k, static_cast<const char*>(a.k) + ((size_t)b * a.HK + kh) * kb, kb, full);
        bulk_g2s(sb + a.off_q, static_cast<const char*>(a.q) + ((size_t)b * a.HK + kh) * kb, kb, full);
        bulk_g2s(sb + a.off_v,
                 static_cast<const char*>(a.v) + (((size_t)b * a.HV + hv) * a.V + (size_t)vb * VB) * sa,
                 VB * sa, full);
        bulk_g2s(sb + a.off_a, a.a + ((size_t)b * a.HV + hv) * KD, KD * 4, full);
    }

    // u = S (a o k), d = beta (v - u), S <- S Diag(a) + d k^T, o = S (a o q) + d (k . q)
    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb, uint8_t*,
                                   int lane, int wi) {
        if (!m.valid) return;
        const bool bf = a.act_bf16;
        const float* tile = reinterpret_cast<const float*>(sb);
        float k4[4], q4[4];
        load4(sb + a.off_k, lane * 4, bf, k4);
        load4(sb + a.off_q, lane * 4, bf, q4);
        const float4 a4 = *reinterpret_cast<const float4*>(sb + a.off_a + lane * 16);
        const float ak[4] = {a4.x * k4[0], a4.y * k4[1], a4.z * k4[2], a4.w * k4[3]};
        const float aq[4] = {a4.x * q4[0], a4.y * q4[1], a4.z * q4[2], a4.w * q4[3]};
        float kq = k4[0] * q4[0] + k4[1] * q4[1] + k4[2] * q4[2] + k4[3] * q4[3];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) kq += __shfl_xor_sync(kFull, kq, o);
        float* dst = a.state + (((size_t)m.s * a.HV + m.hv) * a.V + (size_t)m.vb * VB) * KD;
        const int r0 = wi * RW;
        float part[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float4 s4 = *reinterpret_cast<const float4*>(tile + (r0 + j) * KD + lane * 4);
            part[j] = s4.x * ak[0] + s4.y * ak[1] + s4.z * ak[2] + s4.w * ak[3];
            part[16 + j] = s4.x * aq[0] + s4.y * aq[1] + s4.z * aq[2] + s4.w * aq[3];
        }
        reduce_scatter<32, 32>(part);
        const float cdot = __shfl_down_sync(kFull, part[0], 16);
        float dn = 0.f;
        if (lane < 16) {
            const int r = r0 + lane;
            dn = m.beta * (load1(sb + a.off_v, r, bf) - part[0]);
            const float oo = fmaf(dn, kq, cdot);
            store1(a.o, ((size_t)m.b * a.HV + m.hv) * a.V + (size_t)m.vb * VB + r, a.out_bf16, oo);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float dj = __shfl_sync(kFull, dn, j);
            float4 s4 = *reinterpret_cast<const float4*>(tile + (r0 + j) * KD + lane * 4);
            s4.x = fmaf(s4.x, a4.x, dj * k4[0]);
            s4.y = fmaf(s4.y, a4.y, dj * k4[1]);
            s4.z = fmaf(s4.z, a4.z, dj * k4[2]);
            s4.w = fmaf(s4.w, a4.w, dj * k4[3]);
            *reinterpret_cast<float4*>(dst + (r0 + j) * KD + lane * 4) = s4;
        }
    }
};

}  // namespace kda
}  // namespace rssm

using namespace rssm;

extern "C" size_t rssm_kda_workspace_size(const rssm_gdn_dims* d) {
    if (kda::check_dims(d)) return 0;
    return (kda::kg_offset_floats(d) + (size_t)d->batch * d->num_v_heads * d->ring_len * kda::KD) *
           sizeof(float);
}

extern "C" int rssm_kda_prepare(const rssm_gdn_dims* d, const void* q, const void* k,
                                const float* a, const float* beta, const int32_t* cache_indices,
                                const int32_t* row_wp, const uint8_t* row_flush, void* ring_k,
                                float* ring_a, void* workspace, size_t workspace_bytes,
                                int32_t* dev_err, rssm_stream_t stream) {
    int rc = kda::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(a) || !ok_ptr(beta) || !ok_ptr(cache_indices) ||
        !ok_ptr(row_wp) || !ok_ptr(row_flush) || !ok_ptr(ring_k) || !ok_ptr(ring_a) ||
        !ok_ptr(workspace))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_kda_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    kda::PreArgs pa{};
    pa.q = q; pa.k = k; pa.a = a; pa.beta = beta; pa.ci = cache_indices; pa.row_wp = row_wp;
    pa.row_flush = row_flush; pa.ring_k = ring_k; pa.ring_a = ring_a;
    pa.ws = static_cast<float*>(workspace);
    pa.ws_kg = static_cast<float*>(workspace) + kda::kg_offset_floats(d);
    pa.dev_err = dev_err;
    pa.HV = d->num_v_heads; pa.HK = d->num_k_heads; pa.L = d->ring_len;
    pa.num_slots = d->num_slots; pa.act_bf16 = d->act_dtype == RSSM_BF16;
    pa.n_items = d->batch * d->num_v_heads;
    const unsigned blocks = (unsigned)((pa.n_items + kda::kPreWarps - 1) / kda::kPreWarps);
    kda::prepare_kernel<<<blocks, 32 * kda::kPreWarps, 0, (cudaStream_t)stream>>>(pa);
    return launch_status();
}

extern "C" int rssm_kda_output(const rssm_gdn_dims* d, float* state, const void* v, float* ring_d,
                               const int32_t* cache_indices, const int32_t* row_wp,
                               const uint8_t* row_flush, const void* workspace,
                               size_t workspace_bytes, void* o, int32_t* dev_err,
                               rssm_stream_t stream) {
    int rc = kda::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(v) || !ok_ptr(ring_d) || !ok_ptr(cache_indices) ||
        !ok_ptr(row_wp) || !ok_ptr(row_flush) || !ok_ptr(workspace) || !ok_ptr(o))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_kda_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    kda::OutPolicy::Args a{};
    a.state = state; a.v = v; a.ring_d = ring_d; a.ci = cache_indices; a.row_wp = row_wp;
    a.row_flush = row_flush; a.ws = static_cast<const float*>(workspace);
    a.ws_kg = static_cast<const float*>(workspace) + kda::kg_offset_floats(d);
    a.o = o; a.dev_err = dev_err;
    a.batch = d->batch; a.HV = d->num_v_heads; a.V = d->head_v_dim; a.L = d->ring_len;
    a.num_slots = d->num_slots; a.act_bf16 = d->act_dtype == RSSM_BF16;
    a.out_bf16 = d->out_dtype == RSSM_BF16;
    const int sa = a.act_bf16 ? 2 : 4;
    int off = kda::TILE;
    a.off_vec = off; off += kda::main_floats(a.L) * 4;
    a.off_v = off;   off += (kda::VB * sa + 15) & ~15;
    a.off_d = off;   off += a.L * kda::VB * 4;
    const int stage_bytes = (off + 127) & ~127;
    return launch_pipe<kda::OutPolicy>(a, stage_bytes, 0, kda::TILE,
                                       (long)d->batch * d->num_v_heads * (d->head_v_dim / kda::VB),
                                       (cudaStream_t)stream);
}

extern "C" int rssm_kda_step(const rssm_gdn_dims* d, int advance, const uint8_t* force_flush,
                             int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush, float* state,
                             const void* q, const void* k, const void* v, const float* beta,
                             const float* a, const int32_t* cache_indices, void* ring_k,
                             float* ring_a, float* ring_d, void* workspace,
                             size_t workspace_bytes, void* o, int32_t* dev_err,
                             rssm_stream_t stream) {
    int rc = kda::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (advance) {
        rc = rssm_advance_cursors(RSSM_CURSOR_STANDARD, slot_wp, nullptr, nullptr, cache_indices,
                                  force_flush, nullptr, d->batch, d->num_slots, d->ring_len, 0,
                                  row_wp, row_flush, dev_err, stream);
        if (rc) return rc;
    }
    rc = rssm_kda_prepare(d, q, k, a, beta, cache_indices, row_wp, row_flush, ring_k, ring_a,
                          workspace, workspace_bytes, dev_err, stream);
    if (rc) return rc;
    return rssm_kda_output(d, state, v, ring_d, cache_indices, row_wp, row_flush, workspace,
                           workspace_bytes, o, dev_err, stream);
}

extern "C" int rssm_kda_full_state_decode(const rssm_gdn_dims* d, float* state, const void* q,
                                          const void* k, const void* v, const float* beta,
                                          const float* a, const int32_t* cache_indices, void* o,
                                          int32_t* dev_err, rssm_stream_t stream) {
    int rc = kda::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(beta) || !ok_ptr(a) ||
        !ok_ptr(cache_indices) || !ok_ptr(o))
        return RSSM_ERR_INVALID_ARG;
    kda::FullPolicy::Args fa{};
    fa.state = state; fa.q = q; fa.k = k; fa.v = v; fa.beta = beta; fa.a = a;
    fa.ci = cache_indices; fa.o = o; fa.dev_err = dev_err;
    fa.batch = d->batch; fa.HV = d->num_v_heads; fa.HK = d->num_k_heads; fa.V = d->head_v_dim;
    fa.num_slots = d->num_slots; fa.act_bf16 = d->act_dtype == RSSM_BF16;
    fa.out_bf16 = d->out_dtype == RSSM_BF16;
    const int sa = fa.act_bf16 ? 2 : 4;
    int off = kda::TILE;
    fa.off_k = off; off += kda::KD * sa;
    fa.off_q = off; off += kda::KD * sa;
    fa.off_v = off; off += (kda::VB * sa + 15) & ~15;
    fa.off_a = off; off += kda::KD * 4;
    const int stage_bytes = (off + 127) & ~127;
    return launch_pipe<kda::FullPolicy>(fa, stage_bytes, 0, kda::TILE,
                                        (long)d->batch * d->num_v_heads * (d->head_v_dim / kda::VB),
                                        (cudaStream_t)stream);
}
