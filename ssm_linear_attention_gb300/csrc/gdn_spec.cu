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
//   prologue_kernel    two kinds of CTA in one grid, independent of each other:
//     fold role        a persistent set of CTAs, first in the grid (they are the
//                      long ones) on four of the six CTA slots of an SM, folds the
//                      (row, value head, 32-row block) tiles of the slots with a
//                      pending fold, dealt evenly: S0 rows in registers (4 threads
//                      per row), the committed entries copied into shared memory
//                      asynchronously while those rows load, cnt sequential
//                      delta-rule updates from ring k, raw v, beta, g; S0 stored.
//     table role       one CTA per (row, key head), on the remaining slots: dot
//                      products of every live key (history and drafts) with the
//                      drafts' keys and queries, products of gates, into a
//                      per-(row, value head) table.
//   verify_kernel<T>   persistent TMA pipeline over (row, value head, 32-row
//                      block) tiles of S0: the 2T dot products per value row,
//                      then the draft chain per row; writes o, the drafts' d and
//                      raw v, and (one item per row and head) the drafts' k, g
//                      and beta into the ring.
// The fold must finish before any draft is written into the ring: with a
// pending fold the drafts land on ring positions whose raw entries the fold
// reads. The table role reads only history entries, which no draft overwrites,
// so it shares the fold's launch; every ring write happens in the verify launch.
#include <type_traits>

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
constexpr int kFoldChunk = 16;  // committed entries staged per pass of the fold
constexpr int kFoldList = 2048;  // fold items owned by one fold CTA, at most (fallback path)
static_assert(kFoldChunk * (KD / 4) % kThreads == 0 && kThreads == kFoldChunk * (VB / 4),
              "fold staging: whole 16-byte chunks per thread");

// table per (row, value head): au[T][L], ao[T][L], Gu[T], Go[T], beta[T], g[T], c, base'
__host__ __device__ inline int tbl_floats(int L, int T) { return (2 * T * L + 4 * T + 2 + 3) & ~3; }

// Workspace: the tables [batch][HV][tbl_floats], then the drafts' keys and queries in
// float32 [batch][HK][2T][KD] (k_0, q_0, k_1, q_1, ...), written by the table CTAs.
inline size_t vec_offset_floats(const rssm_gdn_dims* d, int T) {
    return (size_t)d->batch * d->num_v_heads * tbl_floats(d->ring_len, T);
}
inline size_t workspace_floats(const rssm_gdn_dims* d, int T) {
    return vec_offset_floats(d, T) + (size_t)d->batch * d->num_k_heads * 2 * T * KD;
}

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
// prologue: exact fold + tables
// ----------------------------------------------------------------------------

struct ProArgs {
    float* state;
    const void* q;
    const void* k;
    const float* beta;
    const float* g;
    const void* ring_k;
    const void* ring_v;
    const float* ring_g;
    const float* ring_beta;
    const int32_t* ci;
    const int32_t* slot_wp;
    const int32_t* slot_base;
    const uint8_t* slot_flush;
    float* ws;
    float* wsv;  // [batch][HK][2T][KD] float32: the drafts' k_j, q_j (interleaved)
    int T, HV, HK, V, L, num_slots, act_bf16;
    int batch;
    int n_items;  // fold work items: batch * HV * V/VB tiles
    int n_pre;    // table CTAs (batch * HK), after the fold CTAs
    int n_fold;   // persistent fold CTAs, first in the grid (they are the long ones)
};

// Shared memory of the fold role (floats): k [16][KD], raw v [16][VB], beta, g in
// float32, then the chunk's keys and values as copied (activation dtype).
__host__ __device__ inline int fold_smem_floats() { return kFoldChunk * (KD + VB + 2) + kFoldChunk * (KD + VB); }

// Shared memory of the table role (floats): KK [L][T], KQ [L][T], gates
// [HV/HK][L], the drafts' k and q [T][2][KD], the history keys [L][KD].
__host__ __device__ inline int pre_smem_floats(int L, int T, int vpk) {
    return ((2 * L * T + vpk * L + 3) & ~3) + 2 * T * KD + L * KD;
}

// Exact fold of one (row, value head, 32-row block) tile. Thread t owns row t/4
// and the 4-column chunks q, q+4, ..., q+28 (q = t%4) of it, so a row's dot
// product needs two shuffles; the committed entries are replayed in order:
// u = S k, d = beta (v - g u), S = g S + d k^T.
__device__ void fold_tile(const ProArgs& a, int item, float* sm) {
    const int NVB = a.V / VB;
    const int b = item / (a.HV * NVB);
    const int rem = item - b * a.HV * NVB;
    const int hv = rem / NVB, vb = rem - (rem / NVB) * NVB;
    const int s = a.ci[b];
    if (s < 0 || s >= a.num_slots) return;  // the verify reports bad slots
    if (!a.slot_flush[s]) return;
    const int cnt = a.slot_wp[s], base = a.slot_base[s];
    if (cnt <= 0 || cnt > a.L || base < 0 || base >= a.L) return;
    const bool bf = a.act_bf16;
    const int sa = bf ? 2 : 4;
    const int L = a.L;
    const int t = threadIdx.x, r = t >> 2, qd = t & 3;
    const int kh = hv / (a.HV / a.HK);
    float* ks = sm;                       // [16][KD]
    float* vs = ks + kFoldChunk * KD;     // [16][VB]
    float* bs = vs + kFoldChunk * VB;     // [16]
    float* gs = bs + kFoldChunk;          // [16]
    float* tile = a.state + (((size_t)s * a.HV + hv) * a.V + (size_t)vb * VB) * KD;
    float2 S2[16];  // chunk u: columns (qd + 4u)*4 .. +3 as two pairs
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const float4 v4 = *reinterpret_cast<const float4*>(tile + r * KD + (qd + 4 * u) * 4);
        S2[2 * u] = make_float2(v4.x, v4.y);
        S2[2 * u + 1] = make_float2(v4.z, v4.w);
    }
    const char* kr = static_cast<const char*>(a.ring_k) + ((size_t)s * a.HK + kh) * L * KD * sa;
    const char* vr = static_cast<const char*>(a.ring_v) + (((size_t)s * a.HV + hv) * L * a.V + (size_t)vb * VB) * sa;
    uint8_t* kraw = reinterpret_cast<uint8_t*>(gs + kFoldChunk);  // [16][KD] as copied
    uint8_t* vraw = kraw + kFoldChunk * KD * 4;                    // [16][VB] as copied
    for (int e0 = 0; e0 < cnt; e0 += kFoldChunk) {
        const int ne = cnt - e0 < kFoldChunk ? cnt - e0 : kFoldChunk;
        __syncthreads();  // the previous chunk (or tile) is no longer read
        // the chunk's keys and raw values by asynchronous copies (no registers, in
        // flight together with the state rows), beta and g into registers
        const int kc16 = KD * sa / 16, vc16 = VB * sa / 16;
        for (int e = t; e < ne * (kc16 + vc16); e += kThreads) {
            if (e < ne * kc16) {
                const int i = e / kc16, c16 = e - i * kc16;
                cp_async16(kraw + (size_t)e * 16, kr + (size_t)((base + e0 + i) % L) * KD * sa + c16 * 16);
            } else {
                const int e2 = e - ne * kc16, i = e2 / vc16, c16 = e2 - i * vc16;
                cp_async16(vraw + (size_t)e2 * 16,
                           vr + (size_t)((base + e0 + i) % L) * a.V * sa + c16 * 16);
            }
        }
        cp_async_commit();
        float bv = 0.f, gv = 0.f;
        if (t < ne) {
            const int pos = (base + e0 + t) % L;
            bv = a.ring_beta[((size_t)s * a.HV + hv) * L + pos];
            gv = a.ring_g[((size_t)s * a.HV + hv) * L + pos];
        }
        cp_async_wait_all();
        __syncthreads();
        for (int e = t; e < ne * (KD + VB) / 4; e += kThreads) {  // float32 copies
            float f[4];
            if (e < ne * KD / 4) {
                load4(kraw, e * 4, bf, f);
                *reinterpret_cast<float4*>(ks + e * 4) = make_float4(f[0], f[1], f[2], f[3]);
            } else {
                const int e2 = e - ne * KD / 4;
                load4(vraw, e2 * 4, bf, f);
                *reinterpret_cast<float4*>(vs + e2 * 4) = make_float4(f[0], f[1], f[2], f[3]);
            }
        }
        if (t < ne) {
            bs[t] = bv;
            gs[t] = gv;
        }
        __syncthreads();
        for (int i = 0; i < ne; ++i) {
            // the dot and the update run as packed two-wide float32 FMAs over column
            // pairs; the key chunks are read again for the update (fewer registers)
            const float* ki = ks + i * KD + qd * 4;
            float2 pa = make_float2(0.f, 0.f), pb = pa, pc = pa, pd = pa;
#pragma unroll
            for (int u = 0; u < 8; u += 2) {
                const float4 ka = *reinterpret_cast<const float4*>(ki + 16 * u);
                const float4 kb = *reinterpret_cast<const float4*>(ki + 16 * (u + 1));
                pa = __ffma2_rn(S2[2 * u], make_float2(ka.x, ka.y), pa);
                pb = __ffma2_rn(S2[2 * u + 1], make_float2(ka.z, ka.w), pb);
                pc = __ffma2_rn(S2[2 * u + 2], make_float2(kb.x, kb.y), pc);
                pd = __ffma2_rn(S2[2 * u + 3], make_float2(kb.z, kb.w), pd);
            }
            float part = ((pa.x + pa.y) + (pb.x + pb.y)) + ((pc.x + pc.y) + (pd.x + pd.y));
            part += __shfl_xor_sync(kFull, part, 1);
            part += __shfl_xor_sync(kFull, part, 2);
            const float ge = gs[i];
            const float dn = bs[i] * (vs[i * VB + r] - ge * part);
            const float2 g2 = make_float2(ge, ge), d2 = make_float2(dn, dn);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float4 k4 = *reinterpret_cast<const float4*>(ki + 16 * u);
                S2[2 * u] = __ffma2_rn(g2, S2[2 * u], __fmul2_rn(d2, make_float2(k4.x, k4.y)));
                S2[2 * u + 1] = __ffma2_rn(g2, S2[2 * u + 1], __fmul2_rn(d2, make_float2(k4.z, k4.w)));
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
        *reinterpret_cast<float4*>(tile + r * KD + (qd + 4 * u) * 4) =
            make_float4(S2[2 * u].x, S2[2 * u].y, S2[2 * u + 1].x, S2[2 * u + 1].y);
}

// Tables of one (row, key head): the dot products of every live key (history,
// then drafts) with the drafts' keys and queries, then, per value head of this
// key head and draft j (m = history + j):
//   ao_i = prod_{l=i+1..m} gate_l (k_i . q_j), i <= m
//   au_i = prod_{l=i+1..m-1} gate_l (k_i . k_j), i < m
//   Gu = prod_{l<m} gate_l, Go = prod_{l<=m} gate_l, beta_j, g_j.
template <int T>
__device__ void pre_head(const ProArgs& a, int idx, float* sm) {
    constexpr int NV = 2 * T;
    constexpr int NVP = NV <= 2 ? 2 : (NV <= 4 ? 4 : (NV <= 8 ? 8 : 16));
    const int b = idx / a.HK, kh = idx - (idx / a.HK) * a.HK;
    const int s = a.ci[b];
    if (s < 0 || s >= a.num_slots) return;
    const int L = a.L, HV = a.HV, HK = a.HK;
    int c, base_eff;
    if (!history(a.slot_wp[s], a.slot_base[s], a.slot_flush[s], L, T, &c, &base_eff)) return;
    const int nk = c + T;  // live keys: history then drafts
    const int vpk = HV / HK;
    const bool bf = a.act_bf16;
    const int sa = bf ? 2 : 4;
    float* KK = sm;                                   // [L][T]   k_i . k_j
    float* KQ = KK + L * T;                           // [L][T]   k_i . q_j
    float* gts = KQ + L * T;                          // [vpk][L] gates of the live entries
    float* kdq = sm + ((2 * L * T + vpk * L + 3) & ~3);  // [T][2][KD] drafts' k, q
    float* hk = kdq + NV * KD;                           // [c][KD] history keys
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = blockDim.x >> 5;

    // every load is issued before any shared-memory store (one round trip)
    const char* kr = static_cast<const char*>(a.ring_k) + ((size_t)s * HK + kh) * L * KD * sa;
    constexpr int DU = (NV * (KD / 4) + kThreads - 1) / kThreads;  // draft chunks per thread
    constexpr int HU = 16 * (KD / 4) / kThreads;  // history chunks held in registers (c <= 16)
    float dv[DU][4];
#pragma unroll
    for (int u = 0; u < DU; ++u) {
        const int e = t + u * kThreads;
        if (e < NV * (KD / 4)) {
            const int jv = e / (KD / 4), c4 = e - (e / (KD / 4)) * (KD / 4);
            const void* src = (jv & 1) ? a.q : a.k;
            load4(static_cast<const char*>(src) + (((size_t)b * T + (jv >> 1)) * HK + kh) * KD * sa,
                  c4 * 4, bf, dv[u]);
        }
    }
    float hv4[HU][4];
    const int hn = c * (KD / 4);
#pragma unroll
    for (int u = 0; u < HU; ++u) {
        const int e = t + u * kThreads;
        if (e < hn) {
            const int i = e / (KD / 4), c4 = e - (e / (KD / 4)) * (KD / 4);
            load4(kr + (size_t)((base_eff + i) % L) * KD * sa, c4 * 4, bf, hv4[u]);
        }
    }
    for (int e = t + HU * kThreads; e < hn; e += kThreads) {  // long rings: the rest directly
        const int i = e / (KD / 4), c4 = e - (e / (KD / 4)) * (KD / 4);
        float f[4];
        load4(kr + (size_t)((base_eff + i) % L) * KD * sa, c4 * 4, bf, f);
        *reinterpret_cast<float4*>(hk + i * KD + c4 * 4) = make_float4(f[0], f[1], f[2], f[3]);
    }
    for (int x = t; x < vpk * nk; x += blockDim.x) {
        const int hl = x / nk, m = x - (x / nk) * nk, hv = kh * vpk + hl;
        gts[hl * L + m] = m < c ? a.ring_g[((size_t)s * HV + hv) * L + (base_eff + m) % L]
                                : a.g[((size_t)b * T + (m - c)) * HV + hv];
    }
    float* gv = a.wsv + ((size_t)b * HK + kh) * NV * KD;  // the verify's float32 copy
#pragma unroll
    for (int u = 0; u < DU; ++u) {
        const int e = t + u * kThreads;
        if (e < NV * (KD / 4)) {
            const float4 f4 = make_float4(dv[u][0], dv[u][1], dv[u][2], dv[u][3]);
            *reinterpret_cast<float4*>(kdq + e * 4) = f4;
            reinterpret_cast<float4*>(gv)[e] = f4;
        }
    }
#pragma unroll
    for (int u = 0; u < HU; ++u) {
        const int e = t + u * kThreads;
        if (e < hn) *reinterpret_cast<float4*>(hk + e * 4) = make_float4(hv4[u][0], hv4[u][1], hv4[u][2], hv4[u][3]);
    }
    __syncthreads();

    // a warp per live key: lane holds 4 columns; the 2T dots reduce with one
    // reduce-scatter (entry 2j: k_i . k_j, entry 2j+1: k_i . q_j)
    for (int i = warp; i < nk; i += nwarps) {
        float ki[4];
        {
            const float* src = i < c ? hk + i * KD : kdq + (2 * (i - c)) * KD;
            const float4 v = *reinterpret_cast<const float4*>(src + lane * 4);
            ki[0] = v.x; ki[1] = v.y; ki[2] = v.z; ki[3] = v.w;
        }
        float part[NVP];
#pragma unroll
        for (int d = 0; d < NVP; ++d) {
            part[d] = 0.f;
            if (d < NV) {
                const float4 v = *reinterpret_cast<const float4*>(kdq + d * KD + lane * 4);
                part[d] = ki[0] * v.x + ki[1] * v.y + ki[2] * v.z + ki[3] * v.w;
            }
        }
        const int e = reduce_scatter<NVP, 32>(part);
        if ((lane & (32 / NVP - 1)) == 0 && e < NV) {
            if (e & 1) KQ[i * T + (e >> 1)] = part[0];
            else KK[i * T + (e >> 1)] = part[0];
        }
    }
    __syncthreads();

    const int TB = tbl_floats(L, T);
    for (int x = t; x < vpk * T; x += blockDim.x) {
        const int hl = x / T, j = x - (x / T) * T, hv = kh * vpk + hl;
        float* tb = a.ws + ((size_t)b * HV + hv) * TB;
        const float* gl = gts + hl * L;
        const int m = c + j;
        float* au = tb + j * L;
        float* ao = tb + T * L + j * L;
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
        tb[2 * T * L + j] = pk;
        tb[2 * T * L + T + j] = pq;
        tb[2 * T * L + 2 * T + j] = a.beta[((size_t)b * T + j) * HV + hv];
        tb[2 * T * L + 3 * T + j] = a.g[((size_t)b * T + j) * HV + hv];
        if (j == 0) {
            tb[2 * T * L + 4 * T] = __int_as_float(c);
            tb[2 * T * L + 4 * T + 1] = __int_as_float(base_eff);
        }
    }
}

// Fold role (CTA f of the n_fold fold CTAs). Every fold CTA builds the same
// ascending list of the rows with a pending fold (ballots over the batch, one pass
// per kThreads rows), and the list's tiles are dealt round-robin over the fold
// CTAs, so each folds an even share. Batches larger than the list fall back to each CTA checking its own
// items (it = f mod n_fold) and folding the flagged ones.
constexpr int kFoldRowList = 2048;

__device__ void fold_role(const ProArgs& a, int f, float* sm) {
    __shared__ int rows[kFoldRowList];
    __shared__ int wsum[kThreads / 32];
    __shared__ int nrows;
    const int NVB = a.V / VB, per_row = a.HV * NVB;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    if (a.batch <= kFoldRowList) {
        int base = 0;
        for (int b0 = 0; b0 < a.batch; b0 += kThreads) {
            const int b = b0 + t;
            bool flag = false;
            if (b < a.batch) {
                const int s = a.ci[b];
                flag = s >= 0 && s < a.num_slots && a.slot_flush[s];
            }
            const unsigned m = __ballot_sync(0xffffffffu, flag);
            if (lane == 0) wsum[warp] = __popc(m);
            __syncthreads();
            int off = base;
            for (int w = 0; w < warp; ++w) off += wsum[w];
            if (flag) rows[off + __popc(m & ((1u << lane) - 1u))] = b;
            int total = 0;
            for (int w = 0; w < kThreads / 32; ++w) total += wsum[w];
            base += total;
            __syncthreads();
        }
        const int tiles = base * per_row;
        for (int x = f; x < tiles; x += a.n_fold) {
            const int ri = x / per_row;
            fold_tile(a, rows[ri] * per_row + (x - ri * per_row), sm);
        }
        return;
    }
    if (t == 0) nrows = 0;
    __syncthreads();
    for (int it = f + t * a.n_fold; it < a.n_items; it += kThreads * a.n_fold) {
        const int s = a.ci[it / per_row];
        if (s >= 0 && s < a.num_slots && a.slot_flush[s]) rows[atomicAdd(&nrows, 1)] = it;
    }
    __syncthreads();
    const int n = nrows;
    for (int j = 0; j < n; ++j) fold_tile(a, rows[j], sm);
}

template <int T>
__global__ void __launch_bounds__(kThreads, 6) prologue_kernel(const ProArgs a) {
    extern __shared__ __align__(16) float psm[];
    if ((int)blockIdx.x < a.n_fold) fold_role(a, blockIdx.x, psm);
    else pre_head<T>(a, blockIdx.x - a.n_fold, psm);
}

// ----------------------------------------------------------------------------
// verify (warp-specialised pipeline, two consumer warps per tile)
// ----------------------------------------------------------------------------

constexpr int kGroupWarps = 2;
constexpr int RW = VB / kGroupWarps;              // value rows per warp
constexpr int kWarpScratch = 2 * kMaxT * RW * 4;  // W [2T][RW]: S0 . k_j, S0 . q_j

template <int T, bool BF>
struct VerPolicy {
    static constexpr int kGroup = kGroupWarps;
    static constexpr int NV = 2 * T;  // vectors k_0, q_0, k_1, q_1, ...
    static constexpr int NG = (NV + 7) / 8;
    static constexpr int NVP = NV <= 2 ? 2 : (NV <= 4 ? 4 : 8);
    struct Args {
        const float* state;
        const void* q;
        const void* k;
        const void* v;
        float* ring_d;
        void* ring_v;
        void* ring_k;
        float* ring_g;
        float* ring_beta;
        const int32_t* ci;
        const int32_t* slot_wp;
        const int32_t* slot_base;
        const uint8_t* slot_flush;
        const float* ws;
        const float* wsv;  // the drafts' k_j, q_j in float32, from the prologue
        void* o;
        int32_t* dev_err;
        int batch, HV, HK, V, L, num_slots, act_bf16, out_bf16;
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
            if (!history(a.slot_wp[s], a.slot_base[s], a.slot_flush[s], a.L, T, &c, &be)) c = -1;
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
        const int L = a.L;
        constexpr int sa = BF ? 2 : 4;
        const int kh = hv / (a.HV / a.HK);
        const int TB = tbl_floats(L, T);
        constexpr uint32_t vb4 = NV * KD * 4;  // the 2T float32 vectors
        mbar_arrive_expect_tx(full, TILE + vb4 + T * VB * sa + m.c * VB * 4 + TB * 4);
        bulk_g2s_hint(sb, a.state + (((size_t)m.s * a.HV + hv) * a.V + (size_t)vb * VB) * KD, TILE,
                      full, pol);
        bulk_g2s(sb + a.off_kq, a.wsv + ((size_t)b * a.HK + kh) * NV * KD, vb4, full);
        for (int j = 0; j < T; ++j) {
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
        constexpr bool bf = BF;
        constexpr int sa = BF ? 2 : 4;
        const int L = a.L, c = m.c;
        const float* tw = reinterpret_cast<const float*>(sb) + wi * RW * KD;  // this warp's rows
        const float* kqf = reinterpret_cast<const float*>(sb + a.off_kq);  // [2T][KD] float32
        float* W = reinterpret_cast<float*>(scratch);  // [2T][RW]

        // phase A: W[d][row] = S0_row . vec_d. Lane (rg, cg) = (lane/8, lane%8) owns
        // rows rg + 4i (i < 4) and the 4-column chunks at cg*4 + 32u (u < 4): within
        // each quarter-warp the 16-byte shared loads touch 32 distinct banks, and the
        // sums reduce across the 8 lanes of a row group. The products run as packed
        // two-wide float32 FMAs over column pairs (even and odd columns accumulate
        // separately and are added at the end).
        const int cg = lane & 7, rg = lane >> 3;
#pragma unroll
        for (int g8 = 0; g8 < NG; ++g8) {
            float2 acc2[4][NVP];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int d = 0; d < NVP; ++d) acc2[i][d] = make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int col = cg * 4 + 32 * u;
                float4 vv[NVP];
#pragma unroll
                for (int d = 0; d < NVP; ++d) {
                    if (g8 * 8 + d < NV)
                        vv[d] = *reinterpret_cast<const float4*>(kqf + (g8 * 8 + d) * KD + col);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 s4 = *reinterpret_cast<const float4*>(tw + (rg + 4 * i) * KD + col);
                    const float2 slo = make_float2(s4.x, s4.y), shi = make_float2(s4.z, s4.w);
#pragma unroll
                    for (int d = 0; d < NVP; ++d) {
                        if (g8 * 8 + d < NV) {
                            acc2[i][d] = __ffma2_rn(slo, make_float2(vv[d].x, vv[d].y), acc2[i][d]);
                            acc2[i][d] = __ffma2_rn(shi, make_float2(vv[d].z, vv[d].w), acc2[i][d]);
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float acc[NVP];
#pragma unroll
                for (int d = 0; d < NVP; ++d) acc[d] = acc2[i][d].x + acc2[i][d].y;
                const int e = g8 * 8 + reduce_scatter<NVP, 8>(acc);
                if ((cg & (8 / NVP - 1)) == 0 && e < NV) W[e * RW + rg + 4 * i] = acc[0];
            }
        }
        __syncwarp();

        // phase B: the draft chain. Lanes r and r+16 share value row r of this warp:
        // each sums half of the history (even / odd entries), then both run the
        // chain; the low lane stores o, the high lane the drafts' d and raw v.
        const float* tb = reinterpret_cast<const float*>(sb + a.off_tbl);
        const float* dh = reinterpret_cast<const float*>(sb + a.off_d);
        const int r = lane & 15, h = lane >> 4;
        const int rr = wi * RW + r;  // row within the tile
        const size_t vi = (size_t)m.vb * VB + rr;
        float hu[T], ho[T];
#pragma unroll
        for (int j = 0; j < T; ++j) hu[j] = ho[j] = 0.f;
        for (int i = h; i < c; i += 2) {
            const float di = dh[i * VB + rr];
#pragma unroll
            for (int j = 0; j < T; ++j) {
                hu[j] = fmaf(tb[j * L + i], di, hu[j]);
                ho[j] = fmaf(tb[T * L + j * L + i], di, ho[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < T; ++j) {
            hu[j] += __shfl_xor_sync(kFull, hu[j], 16);
            ho[j] += __shfl_xor_sync(kFull, ho[j], 16);
        }
        const float* ex = tb + 2 * T * L;  // Gu[T], Go[T], beta[T], g[T]
        // the chain itself (the dependent part) first, the stores after it
        float dd[T], oo[T], vr[T];
#pragma unroll
        for (int j = 0; j < T; ++j) {
            const float* au = tb + j * L + c;          // au over the drafts' entries
            const float* ao = tb + T * L + j * L + c;
            float u = fmaf(ex[j], W[(2 * j) * RW + r], hu[j]);
            float o_ = fmaf(ex[T + j], W[(2 * j + 1) * RW + r], ho[j]);
#pragma unroll
            for (int jj = 0; jj < j; ++jj) {
                u = fmaf(au[jj], dd[jj], u);
                o_ = fmaf(ao[jj], dd[jj], o_);
            }
            vr[j] = load1(sb + a.off_v + j * VB * sa, rr, bf);
            const float dn = ex[2 * T + j] * (vr[j] - ex[3 * T + j] * u);
            dd[j] = dn;
            oo[j] = fmaf(ao[j], dn, o_);
        }
        // lane half 0 stores o, half 1 the drafts' d and raw v into the ring (positions
        // base' + c + j, wrapping). When o and raw v share a dtype, one store serves
        // both halves.
        const size_t o0 = (((size_t)m.b * T) * a.HV + m.hv) * a.V + vi, ostep = (size_t)a.HV * a.V;
        float* rd = a.ring_d + (((size_t)m.s * a.HV + m.hv) * (a.V / VB) + m.vb) * L * VB + rr;
        const size_t v0 = ((size_t)m.s * a.HV + m.hv) * L * a.V + vi;
        const bool same = (a.out_bf16 != 0) == BF;
        int pos = m.base_eff + c;
        pos -= pos >= L ? L : 0;
#pragma unroll
        for (int j = 0; j < T; ++j) {
            if (same) {
                const size_t e = h ? v0 + (size_t)pos * a.V : o0 + j * ostep;
                store1(h ? a.ring_v : a.o, (long)e, bf, h ? vr[j] : oo[j]);
            } else if (h == 0) {
                store1(a.o, (long)(o0 + j * ostep), a.out_bf16, oo[j]);
            } else {
                store1(a.ring_v, (long)(v0 + (size_t)pos * a.V), bf, vr[j]);
            }
            if (h) rd[pos * VB] = dd[j];
            pos = pos + 1 == L ? 0 : pos + 1;
        }

        // the drafts' g and beta (first tile of each value head) and k (first tile
        // of the first value head of each key head) into the ring
        if (wi == 0 && m.vb == 0) {
            const int pos0 = m.base_eff + c;
            if (lane < T) {
                const int pos = (pos0 + lane) % L;
                a.ring_g[((size_t)m.s * a.HV + m.hv) * L + pos] = ex[3 * T + lane];
                a.ring_beta[((size_t)m.s * a.HV + m.hv) * L + pos] = ex[2 * T + lane];
            }
            const int vpk = a.HV / a.HK;
            if (m.hv % vpk == 0) {
                const int kh = m.hv / vpk;
                constexpr int kc = KD / 4;  // 4-element chunks per key
                for (int x = lane; x < T * kc; x += 32) {
                    const int j = x / kc, part = x - (x / kc) * kc;
                    const int pos = (pos0 + j) % L;
                    const float4 f4 = reinterpret_cast<const float4*>(kqf + (size_t)(2 * j) * KD)[part];
                    char* dst = static_cast<char*>(a.ring_k) + (((size_t)m.s * a.HK + kh) * L + pos) * KD * sa;
                    if (bf) {  // exact: the values came from bf16
                        const uint2 w2 = make_uint2(
                            uint32_t(f_to_bf16(f4.x)) | (uint32_t(f_to_bf16(f4.y)) << 16),
                            uint32_t(f_to_bf16(f4.z)) | (uint32_t(f_to_bf16(f4.w)) << 16));
                        reinterpret_cast<uint2*>(dst)[part] = w2;
                    } else {
                        reinterpret_cast<float4*>(dst)[part] = f4;
                    }
                }
            }
        }
        __syncwarp();
    }
};

}  // namespace spec
}  // namespace rssm

using namespace rssm;

namespace {

template <int T>
int spec_launch(const rssm_gdn_dims* d, float* state, const void* q, const void* k, const void* v,
                const float* beta, const float* g, float* ring_d, void* ring_k, float* ring_g,
                void* ring_v, float* ring_beta, const int32_t* cache_indices,
                const int32_t* slot_wp, const int32_t* slot_base, const uint8_t* slot_flush,
                void* workspace, void* o, int32_t* dev_err, cudaStream_t st) {
    DeviceInfo di;
    if (!device_info(&di)) return RSSM_ERR_CUDA;
    const int HV = d->num_v_heads, HK = d->num_k_heads, V = d->head_v_dim, L = d->ring_len;
    const int NVB = V / spec::VB;
    const bool abf = d->act_dtype == RSSM_BF16;
    const int sa = abf ? 2 : 4;

    // 1. exact fold of slots with a pending fold, and the tables
    int psm = spec::pre_smem_floats(L, T, HV / HK);
    if (psm < spec::fold_smem_floats()) psm = spec::fold_smem_floats();
    const int psmem = psm * 4;
    if (psmem > di.max_smem_optin) return RSSM_ERR_UNSUPPORTED;
    if (psmem > 48 * 1024 &&
        !ensure_smem_limit(reinterpret_cast<const void*>(spec::prologue_kernel<T>), psmem))
        return RSSM_ERR_CUDA;
    spec::ProArgs pa{};
    pa.state = state; pa.q = q; pa.k = k; pa.beta = beta; pa.g = g; pa.ring_k = ring_k;
    pa.ring_v = ring_v; pa.ring_g = ring_g; pa.ring_beta = ring_beta; pa.ci = cache_indices;
    pa.slot_wp = slot_wp; pa.slot_base = slot_base; pa.slot_flush = slot_flush;
    pa.ws = static_cast<float*>(workspace);
    pa.wsv = static_cast<float*>(workspace) + spec::vec_offset_floats(d, T);
    pa.T = T; pa.HV = HV; pa.HK = HK; pa.V = V; pa.L = L; pa.num_slots = d->num_slots;
    pa.act_bf16 = abf;
    pa.batch = d->batch;
    pa.n_items = d->batch * HV * NVB;
    {
        const int per = (pa.n_items + spec::kFoldList - 1) / spec::kFoldList;  // CTAs for <= kFoldList each
        int nf = di.sm_count * 4;  // four of the six CTA slots of an SM; tables fill the rest
        if (nf < per) nf = per;
        if (nf > pa.n_items) nf = pa.n_items;
        pa.n_fold = nf;
    }
    pa.n_pre = d->batch * HK;
    const long blocks = (long)pa.n_fold + pa.n_pre;
    spec::prologue_kernel<T><<<(unsigned)blocks, spec::kThreads, psmem, st>>>(pa);
    if (launch_status()) return RSSM_ERR_CUDA;

    // 2. verify
    const int TBs = spec::tbl_floats(L, T);
    int off = spec::TILE;
    const int off_kq = off; off += 2 * T * spec::KD * 4;
    const int off_v = off;  off += T * spec::VB * sa;
    const int off_d = off;  off += L * spec::VB * 4;
    const int off_tbl = off; off += TBs * 4;
    const int stage_bytes = (off + 127) & ~127;
    auto run = [&](auto* tag) {
        using Pol = std::remove_pointer_t<decltype(tag)>;
        typename Pol::Args va{};
        va.state = state; va.q = q; va.k = k; va.v = v; va.ring_d = ring_d; va.ring_v = ring_v;
        va.ring_k = ring_k; va.ring_g = ring_g; va.ring_beta = ring_beta;
        va.ci = cache_indices; va.slot_wp = slot_wp; va.slot_base = slot_base;
        va.slot_flush = slot_flush; va.ws = static_cast<const float*>(workspace); va.o = o;
        va.wsv = static_cast<const float*>(workspace) + spec::vec_offset_floats(d, T);
        va.dev_err = dev_err; va.batch = d->batch; va.HV = HV; va.HK = HK; va.V = V;
        va.L = L; va.num_slots = d->num_slots; va.act_bf16 = abf;
        va.out_bf16 = d->out_dtype == RSSM_BF16;
        va.off_kq = off_kq; va.off_v = off_v; va.off_d = off_d; va.off_tbl = off_tbl;
        return launch_pipe<Pol>(va, stage_bytes, spec::kWarpScratch, spec::TILE,
                                (long)d->batch * HV * NVB, st);
    };
    if (abf) return run(static_cast<spec::VerPolicy<T, true>*>(nullptr));
    return run(static_cast<spec::VerPolicy<T, false>*>(nullptr));
}

}  // namespace

extern "C" size_t rssm_gdn_spec_workspace_size(const rssm_gdn_dims* d, int32_t T) {
    if (!d || d->batch < 0 || d->num_v_heads <= 0 || d->num_k_heads <= 0 || d->ring_len < 1 ||
        T < 1 || T > spec::kMaxT)
        return 0;
    return spec::workspace_floats(d, T) * sizeof(float);
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
    cudaStream_t st = (cudaStream_t)stream;
#define RSSM_SPEC_CASE(TT)                                                                        \
    case TT:                                                                                      \
        return spec_launch<TT>(d, state, q, k, v, beta, g, ring_d, ring_k, ring_g, ring_v,        \
                               ring_beta, cache_indices, slot_wp, slot_base, slot_flush,          \
                               workspace, o, dev_err, st);
    switch (T) {
        RSSM_SPEC_CASE(1)
        RSSM_SPEC_CASE(2)
        RSSM_SPEC_CASE(3)
        RSSM_SPEC_CASE(4)
        RSSM_SPEC_CASE(5)
        RSSM_SPEC_CASE(6)
        RSSM_SPEC_CASE(7)
        RSSM_SPEC_CASE(8)
        default:
            return RSSM_ERR_UNSUPPORTED;
    }
#undef RSSM_SPEC_CASE
}
