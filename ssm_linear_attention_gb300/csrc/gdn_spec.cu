// gdn_spec.cu -- ReplaySSM speculative verify for the gated delta net (sm_103a).
//
// Pages followed: [SPEC] "[GDN] Support ReplaySSM Ring Spec-Verify" (SGLang PR
// 28695 report): 功能与动机 (the per-draft full-state snapshots of the
// recurrent verify are the bulk of spec-decode memory), 实现拆解 item 2 (ring
// tensors d/k/g plus raw v/k and beta, cursors write_pos / cache_base /
// is_flush per slot), item 3 (gdn_replayssm_spec_circular_kernel reconstructs
// per-draft outputs from the frozen checkpoint + circular ring;
// gdn_replayssm_exact_fold_kernel replays the recurrent update sequentially
// from the raw inputs at a flush), item 4 (the commit only advances cursors),
// 评论区精华 (the exact fold fixed the long-output drift; ring length >= 2 x
// drafts).
//
// Launches of one verify round:
//   fold_kernel        one CTA per (row, value head, 32-row block) of a slot with
//                      a pending fold: S0 rows in registers, the committed entries
//                      staged in shared memory, cnt sequential delta-rule updates
//                      from ring k, raw v, beta, g; S0 stored.
//   spec_pre_kernel    one CTA per (row, key head): dot products of every live key
//                      (history and drafts) with the drafts' keys and queries,
//                      products of gates, into a per-(row, value head) table;
//                      writes the drafts' k, g, beta into the ring.
//   verify_kernel<DP>  persistent TMA pipeline over (row, value head, 32-row
//                      block) tiles of S0: the 2T dot products per value row,
//                      then the draft chain per row; writes o, and d and raw v
//                      of the drafts into the ring.
// A fold must precede the verify in a separate launch: the drafts of the same
// round may land on ring positions whose raw entries the fold still reads.
#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace rssm {
namespace spec {

constexpr int kThreads = 128;
constexpr int KD = 128;
constexpr int VB = 32;  // value rows per work item (a 16 KB fp32 tile)
constexpr int TILE = VB * KD * 4;
constexpr int kMaxT = 8;

// table per (row, value head): au[T][L], ao[T][L], Gu[T], Go[T], beta[T], g[T], c, base'
__host__ __device__ inline int tbl_floats(int L, int T) { return (2 * T * L + 4 * T + 2 + 3) & ~3; }

// Effective history of a slot at verify time: (count, oldest position); false when
// the cursors are outside the ring.
__device__ __forceinline__ bool history(int cnt, int base, int flush, int L, int T, int* c,
                                        int* base_eff) {
    if (cnt < 0 || cnt > L || base < 0 || base >= L) return false;
    if (flush) {
        *c = 0;
        *base_eff = (base + cnt) % L;
    } else {
        *c = cnt;
        *base_eff = base;
    }
    return *c + T <= L;
}

// ----------------------------------------------------------------------------
// exact fold
// ----------------------------------------------------------------------------

struct FoldArgs {
    float* state;
    const void* ring_k;
    const void* ring_v;
    const float* ring_g;
    const float* ring_beta;
    const int32_t* ci;
    const int32_t* slot_wp;
    const int32_t* slot_base;
    const uint8_t* slot_flush;
    int32_t* dev_err;
    int HV, HK, V, L, num_slots, act_bf16;
};

// One CTA (4 warps) per (row, value head, VB-row block) of a slot with a pending
// fold. Warp w owns rows w + 4j (j < VB/4) of the block; a lane holds key columns
// 4l..4l+3 of each, so the block's S0 rows sit in registers. The committed
// entries (k, raw v, beta, g) are staged in shared memory, 16 at a time, then
// replayed in order: u = S k (one reduce-scatter), d = beta (v - g u),
// S = g S + d k^T.
constexpr int kFoldRows = VB / 4;  // rows per warp

__global__ void __launch_bounds__(kThreads) fold_kernel(const FoldArgs a) {
    __shared__ __align__(16) float ks[16 * KD];  // k of up to 16 entries
    __shared__ float vs[16 * VB];                // raw v of the block's rows
    __shared__ float bs[16], gs[16];
    const int NVB = a.V / VB;
    const int item = blockIdx.x;
    const int b = item / (a.HV * NVB);
    const int rem = item - b * a.HV * NVB;
    const int hv = rem / NVB, vb = rem - (rem / NVB) * NVB;
    const int s = a.ci[b];
    if (s < 0 || s >= a.num_slots) return;  // verify reports bad slots
    if (!a.slot_flush[s]) return;
    const int cnt = a.slot_wp[s], base = a.slot_base[s];
    if (cnt <= 0 || cnt > a.L || base < 0 || base >= a.L) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int kh = hv / (a.HV / a.HK);
    float* tile = a.state + (((size_t)s * a.HV + hv) * a.V + (size_t)vb * VB) * KD;
    float S[kFoldRows][4];
#pragma unroll
    for (int j = 0; j < kFoldRows; ++j) {
        const float4 v4 = *reinterpret_cast<const float4*>(tile + (warp + 4 * j) * KD + lane * 4);
        S[j][0] = v4.x; S[j][1] = v4.y; S[j][2] = v4.z; S[j][3] = v4.w;
    }
    constexpr int SH = 32 / kFoldRows;  // lanes holding the same row after the reduce
    for (int e0 = 0; e0 < cnt; e0 += 16) {  // entries in chunks of 16, in order
        const int ne = cnt - e0 < 16 ? cnt - e0 : 16;
        __syncthreads();  // the previous chunk is no longer read
        for (int e = threadIdx.x; e < ne * KD; e += blockDim.x) {
            const int i = e / KD, c = e - (e / KD) * KD;
            const int pos = (base + e0 + i) % a.L;
            ks[e] = load1(a.ring_k, (((size_t)s * a.HK + kh) * a.L + pos) * KD + c, a.act_bf16);
        }
        for (int e = threadIdx.x; e < ne * VB; e += blockDim.x) {
            const int i = e / VB, r = e - (e / VB) * VB;
            const int pos = (base + e0 + i) % a.L;
            vs[e] = load1(a.ring_v, (((size_t)s * a.HV + hv) * a.L + pos) * a.V + (size_t)vb * VB + r,
                          a.act_bf16);
        }
        if (threadIdx.x < ne) {
            const int pos = (base + e0 + threadIdx.x) % a.L;
            bs[threadIdx.x] = a.ring_beta[((size_t)s * a.HV + hv) * a.L + pos];
            gs[threadIdx.x] = a.ring_g[((size_t)s * a.HV + hv) * a.L + pos];
        }
        __syncthreads();
        for (int e = 0; e < ne; ++e) {
            const float4 k4 = *reinterpret_cast<const float4*>(ks + e * KD + lane * 4);
            const float be = bs[e], ge = gs[e];
            float part[kFoldRows];
#pragma unroll
            for (int j = 0; j < kFoldRows; ++j)
                part[j] = S[j][0] * k4.x + S[j][1] * k4.y + S[j][2] * k4.z + S[j][3] * k4.w;
            reduce_scatter<kFoldRows, 32>(part);  // lanes SH*i .. SH*i+SH-1 hold row i's sum
            const int jr = lane / SH;
            const float dmine = be * (vs[e * VB + warp + 4 * jr] - ge * part[0]);
#pragma unroll
            for (int j = 0; j < kFoldRows; ++j) {
                const float dj = __shfl_sync(0xffffffffu, dmine, SH * j);
                S[j][0] = fmaf(ge, S[j][0], dj * k4.x);
                S[j][1] = fmaf(ge, S[j][1], dj * k4.y);
                S[j][2] = fmaf(ge, S[j][2], dj * k4.z);
                S[j][3] = fmaf(ge, S[j][3], dj * k4.w);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kFoldRows; ++j)
        *reinterpret_cast<float4*>(tile + (warp + 4 * j) * KD + lane * 4) =
            make_float4(S[j][0], S[j][1], S[j][2], S[j][3]);
}

// ----------------------------------------------------------------------------
// spec precompute (one CTA per row)
// ----------------------------------------------------------------------------

struct PreArgs {
    const void* q;
    const void* k;
    const float* beta;
    const float* g;
    void* ring_k;
    float* ring_g;
    float* ring_beta;
    const int32_t* ci;
    const int32_t* slot_wp;
    const int32_t* slot_base;
    const uint8_t* slot_flush;
    float* ws;
    int32_t* dev_err;
    int T, HV, HK, L, num_slots, act_bf16;
};

// One CTA per (row, key head): the dot products of every live key (history, then
// drafts) with the drafts' keys and queries, the coefficient tables of the value
// heads that read this key head, and the drafts' ring entries k (this key head),
// g and beta (its value heads).
__global__ void spec_pre_kernel(const PreArgs a) {
    extern __shared__ __align__(16) float psm[];
    const int b = blockIdx.x / a.HK, kh = blockIdx.x - (blockIdx.x / a.HK) * a.HK;
    const int s = a.ci[b];
    if (s < 0 || s >= a.num_slots) return;
    const int T = a.T, L = a.L, HV = a.HV, HK = a.HK;
    int c, base_eff;
    if (!history(a.slot_wp[s], a.slot_base[s], a.slot_flush[s], L, T, &c, &base_eff)) return;
    const int nk = c + T;       // live keys: history then drafts
    const int vpk = HV / HK;
    float* KK = psm;            // [L][T]   k_i . k_j
    float* KQ = KK + L * T;     // [L][T]   k_i . q_j
    float* gts = KQ + L * T;    // [vpk][L] gate of every live entry (history, drafts)
    const int sa = a.act_bf16 ? 2 : 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const char* kin = static_cast<const char*>(a.k);
    const char* qin = static_cast<const char*>(a.q);

    // the drafts' keys and queries, 4 columns per lane, held in registers
    float kd[kMaxT][4], qd[kMaxT][4];
#pragma unroll
    for (int j = 0; j < kMaxT; ++j) {
        if (j < T) {
            load4(kin + (((size_t)b * T + j) * HK + kh) * KD * sa, lane * 4, a.act_bf16, kd[j]);
            load4(qin + (((size_t)b * T + j) * HK + kh) * KD * sa, lane * 4, a.act_bf16, qd[j]);
        }
    }
    for (int i = warp; i < nk; i += nwarps) {
        float ki[4];
        if (i < c) {
            const int pos = (base_eff + i) % L;
            load4(static_cast<const char*>(a.ring_k) + (((size_t)s * HK + kh) * L + pos) * KD * sa,
                  lane * 4, a.act_bf16, ki);
        } else {
            ki[0] = kd[0][0]; ki[1] = kd[0][1]; ki[2] = kd[0][2]; ki[3] = kd[0][3];
#pragma unroll
            for (int j = 1; j < kMaxT; ++j)
                if (j == i - c) { ki[0] = kd[j][0]; ki[1] = kd[j][1]; ki[2] = kd[j][2]; ki[3] = kd[j][3]; }
        }
#pragma unroll
        for (int j = 0; j < kMaxT; ++j) {
            if (j < T) {
                float d1 = ki[0] * kd[j][0] + ki[1] * kd[j][1] + ki[2] * kd[j][2] + ki[3] * kd[j][3];
                float d2 = ki[0] * qd[j][0] + ki[1] * qd[j][1] + ki[2] * qd[j][2] + ki[3] * qd[j][3];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    d1 += __shfl_xor_sync(0xffffffffu, d1, o);
                    d2 += __shfl_xor_sync(0xffffffffu, d2, o);
                }
                if (lane == 0) {
                    KK[i * T + j] = d1;
                    KQ[i * T + j] = d2;
                }
            }
        }
    }
    // gates of the live entries of this key head's value heads, staged once
    for (int x = threadIdx.x; x < vpk * nk; x += blockDim.x) {
        const int hl = x / nk, m = x - (x / nk) * nk, hv = kh * vpk + hl;
        gts[hl * L + m] = m < c ? a.ring_g[((size_t)s * HV + hv) * L + (base_eff + m) % L]
                                : a.g[((size_t)b * T + (m - c)) * HV + hv];
    }
    // the drafts' S-independent ring entries
    const int kc = KD * sa / 16;
    for (int x = threadIdx.x; x < T * kc; x += blockDim.x) {
        const int j = x / kc, part = x - (x / kc) * kc;
        const int pos = (base_eff + c + j) % L;
        reinterpret_cast<uint4*>(static_cast<char*>(a.ring_k) + (((size_t)s * HK + kh) * L + pos) * KD * sa)[part] =
            reinterpret_cast<const uint4*>(kin + (((size_t)b * T + j) * HK + kh) * KD * sa)[part];
    }
    for (int x = threadIdx.x; x < T * vpk; x += blockDim.x) {
        const int j = x / vpk, hv = kh * vpk + (x - (x / vpk) * vpk);
        const int pos = (base_eff + c + j) % L;
        a.ring_g[((size_t)s * HV + hv) * L + pos] = a.g[((size_t)b * T + j) * HV + hv];
        a.ring_beta[((size_t)s * HV + hv) * L + pos] = a.beta[((size_t)b * T + j) * HV + hv];
    }
    __syncthreads();

    // coefficient table per (value head of this key head, draft)
    const int TB = tbl_floats(L, T);
    for (int x = threadIdx.x; x < vpk * T; x += blockDim.x) {
        const int hl = x / T, j = x - (x / T) * T, hv = kh * vpk + hl;
        float* t = a.ws + ((size_t)b * HV + hv) * TB;
        const float* gl = gts + hl * L;
        const int m = c + j;
        float* au = t + j * L;
        float* ao = t + T * L + j * L;
        // ao_i = prod_{l=i+1..m} gate_l * (k_i . q_j), i <= m
        // au_i = prod_{l=i+1..m-1} gate_l * (k_i . k_j), i < m
        float pq = 1.f, pk = 1.f;
        for (int i = m; i >= 0; --i) {
            ao[i] = pq * KQ[i * T + j];
            if (i < m) {
                au[i] = pk * KK[i * T + j];
                pk *= gl[i];
            }
            pq *= gl[i];
        }
        for (int i = m + 1; i < L; ++i) {
            ao[i] = 0.f;
            au[i] = 0.f;
        }
        if (m < L) au[m] = 0.f;
        // pk = prod_{l<m} gate_l (Gu), pq = prod_{l<=m} gate_l (Go)
        t[2 * T * L + j] = pk;
        t[2 * T * L + T + j] = pq;
        t[2 * T * L + 2 * T + j] = a.beta[((size_t)b * T + j) * HV + hv];
        t[2 * T * L + 3 * T + j] = a.g[((size_t)b * T + j) * HV + hv];
        if (j == 0) {
            t[2 * T * L + 4 * T] = __int_as_float(c);
            t[2 * T * L + 4 * T + 1] = __int_as_float(base_eff);
        }
    }
}

// ----------------------------------------------------------------------------
// verify (warp-specialised pipeline, one consumer warp per tile)
// ----------------------------------------------------------------------------

constexpr int kGroupWarps = 2;
constexpr int RW = VB / kGroupWarps;              // value rows per warp
constexpr int kWarpScratch = 3 * kMaxT * RW * 4;  // W [2T][RW] S0 dots, Dd [T][RW] draft d

template <int DP>
struct VerPolicy {
    static constexpr int kGroup = kGroupWarps;
    struct Args {
        const float* state;
        const void* q;
        const void* k;
        const void* v;
        float* ring_d;
        void* ring_v;
        const int32_t* ci;
        const int32_t* slot_wp;
        const int32_t* slot_base;
        const uint8_t* slot_flush;
        const float* ws;
        void* o;
        int32_t* dev_err;
        int batch, T, HV, HK, V, L, num_slots, act_bf16, out_bf16;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
        int off_kq, off_v, off_d, off_tbl;
    };
    struct Meta {
        int valid, s, b, hv, vb, c, base_eff;
    };

    static __device__ int n_items(const Args& a) { return a.batch * a.HV * (a.V / VB); }

    // (slot, history count or -1 when the cursors are bad, oldest position, row)
    static __device__ int4 prefetch(const Args& a, int item) {
        const int b = item / (a.HV * (a.V / VB));
        const int s = a.ci[b];
        int c = 0, be = 0;
        if (s >= 0 && s < a.num_slots) {
            if (!history(a.slot_wp[s], a.slot_base[s], a.slot_flush[s], a.L, a.T, &c, &be)) c = -1;
        }
        return make_int4(s, c, be, b);
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
            if (r.y < 0) set_dev_err(a.dev_err, RSSM_DEVERR_CURSOR);
            else m.valid = 1;
        }
        *meta = m;
        if (!m.valid) {
            mbar_arrive_plain(full);
            return;
        }
        const int T = a.T, L = a.L;
        const int sa = a.act_bf16 ? 2 : 4;
        const int kh = hv / (a.HV / a.HK);
        const int TB = tbl_floats(L, T);
        const uint32_t kb = KD * sa;
        mbar_arrive_expect_tx(full, TILE + 2 * T * kb + T * VB * sa + m.c * VB * 4 + TB * 4);
        bulk_g2s_hint(sb, a.state + (((size_t)m.s * a.HV + hv) * a.V + (size_t)vb * VB) * KD, TILE,
                      full, pol);
        for (int j = 0; j < T; ++j) {
            const size_t src = (((size_t)b * T + j) * a.HK + kh) * kb;
            bulk_g2s(sb + a.off_kq + (2 * j) * kb, static_cast<const char*>(a.k) + src, kb, full);
            bulk_g2s(sb + a.off_kq + (2 * j + 1) * kb, static_cast<const char*>(a.q) + src, kb, full);
            bulk_g2s(sb + a.off_v + j * VB * sa,
                     static_cast<const char*>(a.v) +
                         ((((size_t)b * T + j) * a.HV + hv) * a.V + (size_t)vb * VB) * sa,
                     VB * sa, full);
        }
        // ring d is blocked by 32 value rows; the history entries are at most two runs
        const float* dr = a.ring_d + (((size_t)m.s * a.HV + hv) * NVB + vb) * L * VB;
        const int run1 = m.base_eff + m.c <= L ? m.c : L - m.base_eff;
        if (run1 > 0) bulk_g2s(sb + a.off_d, dr + (size_t)m.base_eff * VB, run1 * VB * 4, full);
        if (m.c > run1) bulk_g2s(sb + a.off_d + run1 * VB * 4, dr, (m.c - run1) * VB * 4, full);
        bulk_g2s(sb + a.off_tbl, a.ws + ((size_t)b * a.HV + hv) * TB, TB * 4, full);
    }

    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb,
                                   uint8_t* scratch, int lane, int wi) {
        if (!m.valid) return;
        constexpr int RC = 32 / DP;  // value rows per reduce-scatter
        const bool bf = a.act_bf16;
        const int sa = bf ? 2 : 4;
        const int T = a.T, L = a.L, c = m.c;
        const int rbase = wi * RW;
        const float* tile = reinterpret_cast<const float*>(sb);
        const uint8_t* kq = sb + a.off_kq;
        float* W = reinterpret_cast<float*>(scratch);  // [2T][RW]
        float* Dd = W + 2 * kMaxT * RW;                // [T][RW]
        // phase A: S0 . k_j and S0 . q_j for this warp's value rows
        float vec[DP][4];
#pragma unroll
        for (int d = 0; d < DP; ++d) {
            if (d < 2 * T) {
                load4(kq + (size_t)d * KD * sa, lane * 4, bf, vec[d]);
            } else {
                vec[d][0] = vec[d][1] = vec[d][2] = vec[d][3] = 0.f;
            }
        }
#pragma unroll 1
        for (int ch = 0; ch < RW / RC; ++ch) {
            float part[32];
#pragma unroll
            for (int jr = 0; jr < RC; ++jr) {
                const float4 s4 =
                    *reinterpret_cast<const float4*>(tile + (rbase + ch * RC + jr) * KD + lane * 4);
#pragma unroll
                for (int d = 0; d < DP; ++d)
                    part[jr * DP + d] =
                        s4.x * vec[d][0] + s4.y * vec[d][1] + s4.z * vec[d][2] + s4.w * vec[d][3];
            }
            reduce_scatter<32, 32>(part);  // lane l holds entry l
            const int jr = lane / DP, d = lane % DP;
            if (d < 2 * T) W[d * RW + ch * RC + jr] = part[0];
        }
        __syncwarp();
        // phase B: the draft chain, one value row per lane
        const float* t = reinterpret_cast<const float*>(sb + a.off_tbl);
        const float* dh = reinterpret_cast<const float*>(sb + a.off_d);
        const int r = rbase + lane;
        const size_t vi = (size_t)m.vb * VB + r;
        for (int j = 0; j < T && lane < RW; ++j) {
            const float* au = t + j * L;
            const float* ao = t + T * L + j * L;
            const int mm = c + j;
            float u = t[2 * T * L + j] * W[(2 * j) * RW + lane];
            float oo = t[2 * T * L + T + j] * W[(2 * j + 1) * RW + lane];
            for (int i = 0; i < c; ++i) {
                const float di = dh[i * VB + r];
                u = fmaf(au[i], di, u);
                oo = fmaf(ao[i], di, oo);
            }
            for (int i = c; i < mm; ++i) {
                const float di = Dd[(i - c) * RW + lane];
                u = fmaf(au[i], di, u);
                oo = fmaf(ao[i], di, oo);
            }
            const float vr = load1(sb + a.off_v + j * VB * sa, r, bf);
            const float dn = t[2 * T * L + 2 * T + j] * (vr - t[2 * T * L + 3 * T + j] * u);
            Dd[j * RW + lane] = dn;
            oo = fmaf(ao[mm], dn, oo);
            const int pos = (m.base_eff + c + j) % L;
            store1(a.o, (((size_t)m.b * T + j) * a.HV + m.hv) * a.V + vi, a.out_bf16, oo);
            a.ring_d[((((size_t)m.s * a.HV + m.hv) * (a.V / VB) + m.vb) * L + pos) * VB + r] = dn;
            store1(a.ring_v, (((size_t)m.s * a.HV + m.hv) * L + pos) * a.V + vi, bf, vr);
        }
        __syncwarp();
    }
};

}  // namespace spec
}  // namespace rssm

using namespace rssm;

extern "C" size_t rssm_gdn_spec_workspace_size(const rssm_gdn_dims* d, int32_t T) {
    if (!d || d->batch < 0 || d->num_v_heads <= 0 || d->ring_len < 1 || T < 1 || T > spec::kMaxT)
        return 0;
    return (size_t)d->batch * d->num_v_heads * spec::tbl_floats(d->ring_len, T) * sizeof(float);
}

extern "C" int rssm_gdn_spec_verify(const rssm_gdn_dims* d, int32_t T, float* state, const void* q,
                                    const void* k, const void* v, const float* beta,
                                    const float* g, float* ring_d, void* ring_k, float* ring_g,
                                    void* ring_v, float* ring_beta, const int32_t* cache_indices,
                                    const int32_t* slot_wp, const int32_t* slot_base,
                                    const uint8_t* slot_flush, void* workspace,
                                    size_t workspace_bytes, void* o, int32_t* dev_err,
                                    rssm_stream_t stream) {
    if (!d) return RSSM_ERR_INVALID_ARG;
    if (d->batch < 0 || d->num_v_heads <= 0 || d->num_k_heads <= 0 || d->head_k_dim <= 0 ||
        d->head_v_dim <= 0 || d->num_slots <= 0 || !ok_dtype(d->act_dtype) || !ok_dtype(d->out_dtype))
        return RSSM_ERR_INVALID_ARG;
    if (d->ring_len < 1 || d->num_v_heads % d->num_k_heads || T < 1 || d->ring_len < 2 * T)
        return RSSM_ERR_CONFIG;
    if (d->head_k_dim != spec::KD || d->head_v_dim % spec::VB || T > spec::kMaxT)
        return RSSM_ERR_UNSUPPORTED;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(beta) || !ok_ptr(g) ||
        !ok_ptr(ring_d) || !ok_ptr(ring_k) || !ok_ptr(ring_g) || !ok_ptr(ring_v) ||
        !ok_ptr(ring_beta) || !ok_ptr(cache_indices) || !ok_ptr(slot_wp) || !ok_ptr(slot_base) ||
        !ok_ptr(slot_flush) || !ok_ptr(workspace) || !ok_ptr(o))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_gdn_spec_workspace_size(d, T)) return RSSM_ERR_INVALID_ARG;
    DeviceInfo di;
    if (!device_info(&di)) return RSSM_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    const int HV = d->num_v_heads, HK = d->num_k_heads, V = d->head_v_dim, L = d->ring_len;
    const int NVB = V / spec::VB;
    const bool abf = d->act_dtype == RSSM_BF16;
    const int sa = abf ? 2 : 4;

    // 1. exact fold of slots with a pending fold
    spec::FoldArgs fa{state, ring_k, ring_v, ring_g, ring_beta, cache_indices, slot_wp, slot_base,
                      slot_flush, dev_err, HV, HK, V, L, d->num_slots, abf};
    spec::fold_kernel<<<d->batch * HV * NVB, spec::kThreads, 0, st>>>(fa);
    if (launch_status()) return RSSM_ERR_CUDA;

    // 2. precompute: key dots, gate products, S-independent ring entries
    const int psmem = (2 * L * T + (HV / HK) * L) * 4;
    if (psmem > di.max_smem_optin) return RSSM_ERR_UNSUPPORTED;
    if (psmem > 48 * 1024 &&
        !ensure_smem_limit(reinterpret_cast<const void*>(spec::spec_pre_kernel), psmem))
        return RSSM_ERR_CUDA;
    spec::PreArgs pa{q, k, beta, g, ring_k, ring_g, ring_beta, cache_indices, slot_wp, slot_base,
                     slot_flush, static_cast<float*>(workspace), dev_err, T, HV, HK, L,
                     d->num_slots, abf};
    spec::spec_pre_kernel<<<d->batch * HK, 128, psmem, st>>>(pa);
    if (launch_status()) return RSSM_ERR_CUDA;

    // 3. verify
    const int TBs = spec::tbl_floats(L, T);
    int off = spec::TILE;
    const int off_kq = off; off += 2 * T * spec::KD * sa;
    const int off_v = off;  off += T * spec::VB * sa;
    const int off_d = off;  off += L * spec::VB * 4;
    const int off_tbl = off; off += TBs * 4;
    const int stage_bytes = (off + 127) & ~127;
    const long items = (long)d->batch * HV * NVB;
    auto fill = [&](auto& va) {
        va.state = state; va.q = q; va.k = k; va.v = v; va.ring_d = ring_d; va.ring_v = ring_v;
        va.ci = cache_indices; va.slot_wp = slot_wp; va.slot_base = slot_base;
        va.slot_flush = slot_flush; va.ws = static_cast<const float*>(workspace); va.o = o;
        va.dev_err = dev_err; va.batch = d->batch; va.T = T; va.HV = HV; va.HK = HK; va.V = V;
        va.L = L; va.num_slots = d->num_slots; va.act_bf16 = abf;
        va.out_bf16 = d->out_dtype == RSSM_BF16;
        va.off_kq = off_kq; va.off_v = off_v; va.off_d = off_d; va.off_tbl = off_tbl;
    };
    if (T <= 1) {
        spec::VerPolicy<2>::Args va{};
        fill(va);
        return launch_pipe<spec::VerPolicy<2>>(va, stage_bytes, spec::kWarpScratch, spec::TILE, items, st);
    }
    if (T <= 2) {
        spec::VerPolicy<4>::Args va{};
        fill(va);
        return launch_pipe<spec::VerPolicy<4>>(va, stage_bytes, spec::kWarpScratch, spec::TILE, items, st);
    }
    if (T <= 4) {
        spec::VerPolicy<8>::Args va{};
        fill(va);
        return launch_pipe<spec::VerPolicy<8>>(va, stage_bytes, spec::kWarpScratch, spec::TILE, items, st);
    }
    spec::VerPolicy<16>::Args va{};
    fill(va);
    return launch_pipe<spec::VerPolicy<16>>(va, stage_bytes, spec::kWarpScratch, spec::TILE, items, st);
}
