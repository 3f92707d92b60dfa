// mamba2.cu -- ReplaySSM decode for Mamba2 on sm_103a.
//
// Pages followed: [M2] "ReplaySSM: cache SSM inputs for faster Mamba2 standard
// decode" (vLLM PR 48018 report): 功能与动机 (decode is memory bound; most
// steps read their output from checkpoint + input buffer, the full state is
// written back once every L steps, halving store traffic), 实现拆解 item 1 (a
// precompute kernel for non-flush rows and an output kernel that branches per
// row on is_flush), 实现拆解 item 2 (x_cache, dt_cache, B_cache), 关键源码片段
// (argument lists of the ReplaySSM call and of the baseline
// selective_state_update).
//
// Kernels:
//   ring_append_kernel    one CTA per row: x, dt = softplus(dt_raw + dt_bias), B
//                         into ring entry w.
//   precompute_kernel     one CTA per row: B_i . C_t per group, decay suffix
//                         products per head, written as per-(row, head) tables.
//   output_kernel<P,N,ST> persistent, one work item = one (row, head) checkpoint
//                         tile. A single thread feeds a multi-stage ring of shared
//                         memory buffers with 1-D TMA bulk copies (tile, ring x
//                         entries, C, z, table, and on flush rows the ring B
//                         entries) completing on one mbarrier per stage; 128
//                         threads reduce the tile against C with 16-byte shared
//                         loads and a warp reduce-scatter, and flush rows fold the
//                         ring into the tile in registers and store it.
//   full_state_kernel<P,N,ST>  the conventional step (read tile, update, write
//                         tile, output) on the same pipeline.
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace rssm {
namespace m2 {

constexpr int kThreads = 128;
constexpr int kMaxStages = 8;
constexpr int kFixedSmem = 1024;  // barriers + per-stage metadata, before the stages

__host__ __device__ inline int tbl_floats(int L) { return (2 * L + 1 + 3) & ~3; }

struct Meta {
    int valid, s, b, h, w, f;
    float dt, dA;
};

// ----------------------------------------------------------------------------
// ring append
// ----------------------------------------------------------------------------

__global__ void ring_append_kernel(int H, int P, int N, int G, int L, int num_slots, int act_bf16,
                                   const void* __restrict__ x, const float* __restrict__ dt_raw,
                                   const float* __restrict__ dt_bias, int softplus,
                                   const void* __restrict__ B, const int32_t* __restrict__ ci,
                                   const int32_t* __restrict__ row_wp, void* __restrict__ ring_x,
                                   float* __restrict__ ring_dt, void* __restrict__ ring_B,
                                   int32_t* __restrict__ dev_err) {
    const int b = blockIdx.x;
    const int s = ci[b];
    if (s < 0) return;
    if (s >= num_slots) {
        if (threadIdx.x == 0) set_dev_err(dev_err, RSSM_DEVERR_SLOT);
        return;
    }
    const int w = row_wp[b];
    if (w < 0 || w >= L) {
        if (threadIdx.x == 0) set_dev_err(dev_err, RSSM_DEVERR_CURSOR);
        return;
    }
    const int sa = act_bf16 ? 2 : 4;
    const int xc = P * sa / 16;  // 16-byte chunks per head row
    const uint4* xs = reinterpret_cast<const uint4*>(static_cast<const char*>(x) + (size_t)b * H * P * sa);
    for (int c = threadIdx.x; c < H * xc; c += blockDim.x) {
        const int h = c / xc, j = c % xc;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(ring_x) +
                                              (((size_t)s * H + h) * L + w) * P * sa) + j;
        *dst = xs[c];
    }
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        float v = dt_raw[(size_t)b * H + h] + (dt_bias ? dt_bias[h] : 0.f);
        if (softplus) v = softplus_f(v);
        ring_dt[((size_t)s * H + h) * L + w] = v;
    }
    const int bc = N * sa / 16;
    const uint4* bs = reinterpret_cast<const uint4*>(static_cast<const char*>(B) + (size_t)b * G * N * sa);
    for (int c = threadIdx.x; c < G * bc; c += blockDim.x) {
        const int g = c / bc, j = c % bc;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(ring_B) +
                                              (((size_t)s * G + g) * L + w) * N * sa) + j;
        *dst = bs[c];
    }
}

// ----------------------------------------------------------------------------
// precompute: per-(row, head) coefficient tables
// ----------------------------------------------------------------------------

__global__ void precompute_kernel(int H, int N, int G, int L, int num_slots, int act_bf16,
                                  const float* __restrict__ A, const void* __restrict__ C,
                                  const float* __restrict__ ring_dt, const void* __restrict__ ring_B,
                                  const int32_t* __restrict__ ci, const int32_t* __restrict__ row_wp,
                                  float* __restrict__ ws) {
    extern __shared__ __align__(16) float psm[];
    const int b = blockIdx.x;
    const int s = ci[b];
    if (s < 0 || s >= num_slots) return;  // the output kernel reports bad slots
    const int w = row_wp[b];
    if (w < 0 || w >= L) return;
    const int TBL = tbl_floats(L);
    const int bc_len = (G * L + 3) & ~3;
    float* bc = psm;           // [G][L]
    float* tbl = psm + bc_len;  // [H][TBL]
    const int sa = act_bf16 ? 2 : 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;

    // B_i . C_t for every group and live entry i = 0..w
    for (int pair = warp; pair < G * (w + 1); pair += nwarps) {
        const int g = pair / (w + 1), i = pair % (w + 1);
        const char* Bi = static_cast<const char*>(ring_B) + (((size_t)s * G + g) * L + i) * N * sa;
        const char* Ct = static_cast<const char*>(C) + ((size_t)b * G + g) * N * sa;
        float acc = 0.f;
        for (int n = lane; n < N; n += 32) acc += load1(Bi, n, act_bf16) * load1(Ct, n, act_bf16);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) bc[g * L + i] = acc;
    }
    __syncthreads();

    // P_i = exp(A_h * sum_{j>i} dt_j); coef_i = P_i dt_i bc_i; a_i = P_i dt_i; Pm1
    const int hpg = H / G;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const int g = h / hpg;
        const float* dts = ring_dt + ((size_t)s * H + h) * L;
        float* t = tbl + h * TBL;
        const float Ah = A[h];
        float suffix = 0.f;
        for (int i = w; i >= 0; --i) {
            const float dti = dts[i];
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
    __syncthreads();
    float4* dst = reinterpret_cast<float4*>(ws + (size_t)b * H * TBL);
    const float4* src = reinterpret_cast<const float4*>(tbl);
    for (int c = threadIdx.x; c < H * TBL / 4; c += blockDim.x) dst[c] = src[c];
}

// ----------------------------------------------------------------------------
// persistent streaming kernels
// ----------------------------------------------------------------------------

struct OutArgs {
    void* state;
    const void* C;
    const float* D;
    const void* z;
    const void* ring_x;
    const void* ring_B;
    const int32_t* ci;
    const int32_t* row_wp;
    const uint8_t* row_flush;
    const float* ws;
    void* y;
    int32_t* dev_err;
    int batch, H, G, L, num_slots, act_bf16, out_bf16;
    int stages, stage_bytes;
    int off_x, off_C, off_z, off_tbl, off_B;
};

struct FullArgs {
    void* state;
    const void* x;
    const float* dt_raw;
    const float* dt_bias;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const int32_t* ci;
    void* y;
    int32_t* dev_err;
    int batch, H, G, num_slots, act_bf16, out_bf16, softplus;
    int stages, stage_bytes;
    int off_x, off_B, off_C, off_z;
};

__device__ __forceinline__ void mbar_arrive_plain(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Row metadata prefetch for the producer thread: one item ahead.
struct RowMeta {
    int b, s, w, f;
};

template <int P, int N, class ST>
__global__ void __launch_bounds__(kThreads) output_kernel(const OutArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    Meta* meta = reinterpret_cast<Meta*>(smem + 128);
    int* abort_flag = reinterpret_cast<int*>(smem + 128 + kMaxStages * sizeof(Meta));
    uint8_t* stage0 = smem + kFixedSmem;

    constexpr int SS = ST::bytes;
    constexpr int TILE = P * N * SS;
    constexpr int NQ = N / 8;             // lanes per state row (8 elements each)
    constexpr int RP = kThreads / NQ;     // rows per pass
    constexpr int KR = P / RP;            // rows per thread
    constexpr int DUP = NQ / KR;          // lanes holding the same reduced row
    static_assert(KR >= 1 && KR <= NQ, "tile shape");

    const int tid = threadIdx.x;
    const int H = a.H, L = a.L, G = a.G;
    const int sa = a.act_bf16 ? 2 : 4;
    const int TBL = tbl_floats(L);
    const int n_items = a.batch * H;
    const int stages = a.stages;

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(&bars[st], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // ---- producer (thread 0) ----
    uint64_t pol = 0;
    RowMeta pf{-1, 0, 0, 0};
    auto load_row = [&](int b) {
        RowMeta r{b, a.ci[b], 0, 0};
        if (r.s >= 0 && r.s < a.num_slots) {
            r.w = a.row_wp[b];
            r.f = a.row_flush[b];
        }
        return r;
    };
    auto issue = [&](int k) {
        const int item = blockIdx.x + k * gridDim.x;
        if (item >= n_items) return;
        const int st = k % stages;
        uint8_t* sb = stage0 + st * a.stage_bytes;
        const int b = item / H, h = item - (item / H) * H;
        const RowMeta r = (pf.b == b) ? pf : load_row(b);
        const int nxt = item + gridDim.x;
        if (nxt < n_items) pf = load_row(nxt / H);
        Meta m;
        m.b = b; m.h = h; m.s = r.s; m.w = r.w; m.f = r.f; m.valid = 0; m.dt = 0.f; m.dA = 0.f;
        if (r.s >= a.num_slots) {
            set_dev_err(a.dev_err, RSSM_DEVERR_SLOT);
        } else if (r.s >= 0) {
            if (r.w < 0 || r.w >= L) set_dev_err(a.dev_err, RSSM_DEVERR_CURSOR);
            else m.valid = 1;
        }
        meta[st] = m;
        if (!m.valid) {
            mbar_arrive_plain(&bars[st]);
            return;
        }
        const int g = h / (H / G);
        const int w = r.w;
        const uint32_t xbytes = (w + 1) * P * sa;
        const uint32_t bbytes = r.f ? (w + 1) * N * sa : 0;
        const uint32_t tx = TILE + xbytes + N * sa + (a.z ? P * sa : 0) + TBL * 4 + bbytes;
        mbar_arrive_expect_tx(&bars[st], tx);
        const char* state = static_cast<const char*>(a.state);
        bulk_g2s_hint(sb, state + ((size_t)r.s * H + h) * TILE, TILE, &bars[st], pol);
        bulk_g2s(sb + a.off_x,
                 static_cast<const char*>(a.ring_x) + ((size_t)r.s * H + h) * L * P * sa, xbytes,
                 &bars[st]);
        bulk_g2s(sb + a.off_C, static_cast<const char*>(a.C) + ((size_t)b * G + g) * N * sa, N * sa,
                 &bars[st]);
        if (a.z)
            bulk_g2s(sb + a.off_z, static_cast<const char*>(a.z) + ((size_t)b * H + h) * P * sa,
                     P * sa, &bars[st]);
        bulk_g2s(sb + a.off_tbl, a.ws + ((size_t)b * H + h) * TBL, TBL * 4, &bars[st]);
        if (r.f)
            bulk_g2s(sb + a.off_B,
                     static_cast<const char*>(a.ring_B) + ((size_t)r.s * G + g) * L * N * sa, bbytes,
                     &bars[st]);
    };
    if (tid == 0) {
        pol = policy_evict_first();
        for (int k = 0; k < stages; ++k) issue(k);
    }

    // ---- consumers (all threads) ----
    const int q = tid % NQ, r0 = tid / NQ;
    int k = 0;
    for (;; ++k) {
        const int item = blockIdx.x + k * gridDim.x;
        if (item >= n_items) break;
        const int st = k % stages;
        const uint32_t par = (k / stages) & 1;
        // all threads agree on the outcome, so the branch below stays uniform
        const bool ok = __syncthreads_and(mbar_wait_bounded(&bars[st], par) ? 1 : 0) != 0;
        if (!ok) {
            *abort_flag = 1;
            set_dev_err(a.dev_err, RSSM_DEVERR_TIMEOUT);
        }
        const Meta m = meta[st];
        if (ok && m.valid) {
            const uint8_t* sb = stage0 + st * a.stage_bytes;
            const float* tbl = reinterpret_cast<const float*>(sb + a.off_tbl);
            const uint8_t* xr = sb + a.off_x;
            float c[8];
            load8(sb + a.off_C + q * 8 * sa, a.act_bf16, c);
            float part[KR];
#pragma unroll
            for (int kk = 0; kk < KR; ++kk) {
                const int p = r0 + RP * kk;
                float s8[8];
                load8(sb + ((size_t)p * N + q * 8) * SS, ST::bf16, s8);
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) acc = fmaf(s8[j], c[j], acc);
                part[kk] = acc;
            }
            const int kidx = reduce_scatter<KR, NQ>(part);
            const float Pm1 = tbl[2 * L];
            const int w = m.w;
            if ((q & (DUP - 1)) == 0) {
                const int p = r0 + RP * kidx;
                float acc = Pm1 * part[0];
                for (int i = 0; i <= w; ++i) acc = fmaf(tbl[i], load1(xr, i * P + p, a.act_bf16), acc);
                acc = fmaf(__ldg(a.D + m.h), load1(xr, w * P + p, a.act_bf16), acc);
                if (a.z) acc *= silu_f(load1(sb + a.off_z, p, a.act_bf16));
                store1(a.y, ((size_t)m.b * H + m.h) * P + p, a.out_bf16, acc);
            }
            if (m.f) {
                // S_new = Pm1 * S0 + sum_{i<=w} a_i x_i B_i^T, stored rounded to the state dtype
                const float* av = tbl + L;
                const uint8_t* br = sb + a.off_B;
                char* dst_tile = static_cast<char*>(a.state) + ((size_t)m.s * H + m.h) * TILE;
                constexpr int RC = KR < 8 ? KR : 8;
#pragma unroll
                for (int kc = 0; kc < KR; kc += RC) {
                    float acc[RC][8];
#pragma unroll
                    for (int r = 0; r < RC; ++r) {
                        const int p = r0 + RP * (kc + r);
                        float s8[8];
                        load8(sb + ((size_t)p * N + q * 8) * SS, ST::bf16, s8);
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[r][j] = Pm1 * s8[j];
                    }
                    for (int i = 0; i <= w; ++i) {
                        float bi[8];
                        load8(br + ((size_t)i * N + q * 8) * sa, a.act_bf16, bi);
                        const float ai = av[i];
#pragma unroll
                        for (int r = 0; r < RC; ++r) {
                            const int p = r0 + RP * (kc + r);
                            const float ax = ai * load1(xr, i * P + p, a.act_bf16);
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[r][j] = fmaf(ax, bi[j], acc[r][j]);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < RC; ++r) {
                        const int p = r0 + RP * (kc + r);
                        store8(dst_tile + ((size_t)p * N + q * 8) * SS, ST::bf16, acc[r]);
                    }
                }
            }
        }
        __syncthreads();
        if (*abort_flag) break;
        if (tid == 0) issue(k + stages);
    }
    // wind down after a timeout: wait (bounded) for copies still in flight
    if (*abort_flag && tid == 0) {
        for (int j = k; j < k + stages; ++j) {
            const int item = blockIdx.x + j * gridDim.x;
            if (item >= n_items) break;
            mbar_wait_bounded(&bars[j % stages], (j / stages) & 1);
        }
    }
}

template <int P, int N, class ST>
__global__ void __launch_bounds__(kThreads) full_state_kernel(const FullArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    Meta* meta = reinterpret_cast<Meta*>(smem + 128);
    int* abort_flag = reinterpret_cast<int*>(smem + 128 + kMaxStages * sizeof(Meta));
    uint8_t* stage0 = smem + kFixedSmem;

    constexpr int SS = ST::bytes;
    constexpr int TILE = P * N * SS;
    constexpr int NQ = N / 8;
    constexpr int RP = kThreads / NQ;
    constexpr int KR = P / RP;
    constexpr int DUP = NQ / KR;

    const int tid = threadIdx.x;
    const int H = a.H, G = a.G;
    const int sa = a.act_bf16 ? 2 : 4;
    const int n_items = a.batch * H;
    const int stages = a.stages;

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(&bars[st], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    uint64_t pol = 0;
    auto issue = [&](int k) {
        const int item = blockIdx.x + k * gridDim.x;
        if (item >= n_items) return;
        const int st = k % stages;
        uint8_t* sb = stage0 + st * a.stage_bytes;
        const int b = item / H, h = item - (item / H) * H;
        const int s = a.ci[b];
        Meta m;
        m.b = b; m.h = h; m.s = s; m.w = 0; m.f = 0; m.valid = 0; m.dt = 0.f; m.dA = 0.f;
        if (s >= a.num_slots) set_dev_err(a.dev_err, RSSM_DEVERR_SLOT);
        else if (s >= 0) m.valid = 1;
        if (m.valid) {
            float dt = a.dt_raw[(size_t)b * H + h] + (a.dt_bias ? a.dt_bias[h] : 0.f);
            if (a.softplus) dt = softplus_f(dt);
            m.dt = dt;
            m.dA = expf(a.A[h] * dt);
        }
        meta[st] = m;
        if (!m.valid) {
            mbar_arrive_plain(&bars[st]);
            return;
        }
        const int g = h / (H / G);
        const uint32_t tx = TILE + P * sa + 2 * N * sa + (a.z ? P * sa : 0);
        mbar_arrive_expect_tx(&bars[st], tx);
        bulk_g2s_hint(sb, static_cast<const char*>(a.state) + ((size_t)s * H + h) * TILE, TILE,
                      &bars[st], pol);
        bulk_g2s(sb + a.off_x, static_cast<const char*>(a.x) + ((size_t)b * H + h) * P * sa, P * sa,
                 &bars[st]);
        bulk_g2s(sb + a.off_B, static_cast<const char*>(a.B) + ((size_t)b * G + g) * N * sa, N * sa,
                 &bars[st]);
        bulk_g2s(sb + a.off_C, static_cast<const char*>(a.C) + ((size_t)b * G + g) * N * sa, N * sa,
                 &bars[st]);
        if (a.z)
            bulk_g2s(sb + a.off_z, static_cast<const char*>(a.z) + ((size_t)b * H + h) * P * sa,
                     P * sa, &bars[st]);
    };
    if (tid == 0) {
        pol = policy_evict_first();
        for (int k = 0; k < stages; ++k) issue(k);
    }

    const int q = tid % NQ, r0 = tid / NQ;
    int k = 0;
    for (;; ++k) {
        const int item = blockIdx.x + k * gridDim.x;
        if (item >= n_items) break;
        const int st = k % stages;
        const uint32_t par = (k / stages) & 1;
        // all threads agree on the outcome, so the branch below stays uniform
        const bool ok = __syncthreads_and(mbar_wait_bounded(&bars[st], par) ? 1 : 0) != 0;
        if (!ok) {
            *abort_flag = 1;
            set_dev_err(a.dev_err, RSSM_DEVERR_TIMEOUT);
        }
        const Meta m = meta[st];
        if (ok && m.valid) {
            const uint8_t* sb = stage0 + st * a.stage_bytes;
            float c[8], bq[8];
            load8(sb + a.off_C + q * 8 * sa, a.act_bf16, c);
            load8(sb + a.off_B + q * 8 * sa, a.act_bf16, bq);
            char* dst_tile = static_cast<char*>(a.state) + ((size_t)m.s * H + m.h) * TILE;
            float part[KR];
#pragma unroll
            for (int kk = 0; kk < KR; ++kk) {
                const int p = r0 + RP * kk;
                float s8[8];
                load8(sb + ((size_t)p * N + q * 8) * SS, ST::bf16, s8);
                const float dx = m.dt * load1(sb + a.off_x, p, a.act_bf16);
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    s8[j] = fmaf(m.dA, s8[j], dx * bq[j]);
                    acc = fmaf(s8[j], c[j], acc);
                }
                part[kk] = acc;
                store8(dst_tile + ((size_t)p * N + q * 8) * SS, ST::bf16, s8);
            }
            const int kidx = reduce_scatter<KR, NQ>(part);
            if ((q & (DUP - 1)) == 0) {
                const int p = r0 + RP * kidx;
                float acc = fmaf(__ldg(a.D + m.h), load1(sb + a.off_x, p, a.act_bf16), part[0]);
                if (a.z) acc *= silu_f(load1(sb + a.off_z, p, a.act_bf16));
                store1(a.y, ((size_t)m.b * H + m.h) * P + p, a.out_bf16, acc);
            }
        }
        __syncthreads();
        if (*abort_flag) break;
        if (tid == 0) issue(k + stages);
    }
    if (*abort_flag && tid == 0) {
        for (int j = k; j < k + stages; ++j) {
            const int item = blockIdx.x + j * gridDim.x;
            if (item >= n_items) break;
            mbar_wait_bounded(&bars[j % stages], (j / stages) & 1);
        }
    }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------

int check_dims(const rssm_mamba2_dims* d) {
    if (!d) return RSSM_ERR_INVALID_ARG;
    if (d->batch < 0 || d->nheads <= 0 || d->headdim <= 0 || d->dstate <= 0 || d->ngroups <= 0 ||
        d->num_slots <= 0)
        return RSSM_ERR_INVALID_ARG;
    if (!ok_dtype(d->state_dtype) || !ok_dtype(d->act_dtype) || !ok_dtype(d->out_dtype))
        return RSSM_ERR_INVALID_ARG;
    if (d->ring_len < 1 || d->nheads % d->ngroups) return RSSM_ERR_CONFIG;
    if ((d->headdim != 64 && d->headdim != 128) || (d->dstate != 64 && d->dstate != 128))
        return RSSM_ERR_UNSUPPORTED;
    return RSSM_OK;
}

template <class F>
int dispatch_pn(int P, int N, int state_dtype, F&& f) {
#define RSSM_M2_CASE(PP, NN)                                                        \
    if (P == PP && N == NN) {                                                        \
        if (state_dtype == RSSM_BF16) return f.template go<PP, NN, StBF16>();        \
        return f.template go<PP, NN, StF32>();                                       \
    }
    RSSM_M2_CASE(64, 128)
    RSSM_M2_CASE(128, 128)
    RSSM_M2_CASE(64, 64)
    RSSM_M2_CASE(128, 64)
#undef RSSM_M2_CASE
    return RSSM_ERR_UNSUPPORTED;
}

struct OutLaunch {
    OutArgs a;
    cudaStream_t stream;
    template <int P, int N, class ST>
    int go() {
        DeviceInfo di;
        if (!device_info(&di)) return RSSM_ERR_CUDA;
        const int sa = a.act_bf16 ? 2 : 4;
        const int L = a.L;
        int off = P * N * ST::bytes;
        a.off_x = off;   off += L * P * sa;
        a.off_C = off;   off += N * sa;
        a.off_z = off;   off += P * sa;
        a.off_tbl = off; off += tbl_floats(L) * 4;
        a.off_B = off;   off += L * N * sa;
        a.stage_bytes = (off + 127) & ~127;
        PipeShape ps;
        if (!pick_pipe_shape(di, a.stage_bytes, kFixedSmem, kMaxStages, &ps)) return RSSM_ERR_UNSUPPORTED;
        a.stages = ps.stages;
        const void* kfn = reinterpret_cast<const void*>(output_kernel<P, N, ST>);
        if (!ensure_smem_limit(kfn, ps.smem_bytes)) return RSSM_ERR_CUDA;
        const long items = (long)a.batch * a.H;
        long grid = (long)di.sm_count * ps.ctas_per_sm;
        if (grid > items) grid = items;
        output_kernel<P, N, ST><<<(int)grid, kThreads, ps.smem_bytes, stream>>>(a);
        return launch_status();
    }
};

struct FullLaunch {
    FullArgs a;
    cudaStream_t stream;
    template <int P, int N, class ST>
    int go() {
        DeviceInfo di;
        if (!device_info(&di)) return RSSM_ERR_CUDA;
        const int sa = a.act_bf16 ? 2 : 4;
        int off = P * N * ST::bytes;
        a.off_x = off; off += P * sa;
        a.off_B = off; off += N * sa;
        a.off_C = off; off += N * sa;
        a.off_z = off; off += P * sa;
        a.stage_bytes = (off + 127) & ~127;
        PipeShape ps;
        if (!pick_pipe_shape(di, a.stage_bytes, kFixedSmem, kMaxStages, &ps)) return RSSM_ERR_UNSUPPORTED;
        a.stages = ps.stages;
        const void* kfn = reinterpret_cast<const void*>(full_state_kernel<P, N, ST>);
        if (!ensure_smem_limit(kfn, ps.smem_bytes)) return RSSM_ERR_CUDA;
        const long items = (long)a.batch * a.H;
        long grid = (long)di.sm_count * ps.ctas_per_sm;
        if (grid > items) grid = items;
        full_state_kernel<P, N, ST><<<(int)grid, kThreads, ps.smem_bytes, stream>>>(a);
        return launch_status();
    }
};

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
    m2::ring_append_kernel<<<d->batch, 256, 0, (cudaStream_t)stream>>>(
        d->nheads, d->headdim, d->dstate, d->ngroups, d->ring_len, d->num_slots,
        d->act_dtype == RSSM_BF16, x, dt_raw, dt_bias, dt_softplus, B, cache_indices, row_wp, ring_x,
        ring_dt, ring_B, dev_err);
    return launch_status();
}

extern "C" size_t rssm_mamba2_workspace_size(const rssm_mamba2_dims* d) {
    if (m2::check_dims(d)) return 0;
    return (size_t)d->batch * d->nheads * m2::tbl_floats(d->ring_len) * sizeof(float);
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
    const int L = d->ring_len;
    const int smem = (((d->ngroups * L + 3) & ~3) + d->nheads * m2::tbl_floats(L)) * 4;
    DeviceInfo di;
    if (!device_info(&di)) return RSSM_ERR_CUDA;
    if (smem > di.max_smem_optin) return RSSM_ERR_UNSUPPORTED;
    if (smem > 48 * 1024 &&
        !ensure_smem_limit(reinterpret_cast<const void*>(m2::precompute_kernel), smem))
        return RSSM_ERR_CUDA;
    m2::precompute_kernel<<<d->batch, 128, smem, (cudaStream_t)stream>>>(
        d->nheads, d->dstate, d->ngroups, L, d->num_slots, d->act_dtype == RSSM_BF16, A, C, ring_dt,
        ring_B, cache_indices, row_wp, static_cast<float*>(workspace));
    return launch_status();
}

extern "C" int rssm_mamba2_output(const rssm_mamba2_dims* d, void* state, const void* C,
                                  const float* D, const void* z, const void* ring_x,
                                  const void* ring_B, const int32_t* cache_indices,
                                  const int32_t* row_wp, const uint8_t* row_flush,
                                  const void* workspace, size_t workspace_bytes, void* y,
                                  int32_t* dev_err, rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(C) || !ok_ptr(D) || !ok_opt_ptr(z) || !ok_ptr(ring_x) ||
        !ok_ptr(ring_B) || !ok_ptr(cache_indices) || !ok_ptr(row_wp) || !ok_ptr(row_flush) ||
        !ok_ptr(workspace) || !ok_ptr(y))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_mamba2_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    m2::OutLaunch l{};
    l.stream = (cudaStream_t)stream;
    m2::OutArgs& a = l.a;
    a.state = state; a.C = C; a.D = D; a.z = z; a.ring_x = ring_x; a.ring_B = ring_B;
    a.ci = cache_indices; a.row_wp = row_wp; a.row_flush = row_flush;
    a.ws = static_cast<const float*>(workspace); a.y = y; a.dev_err = dev_err;
    a.batch = d->batch; a.H = d->nheads; a.G = d->ngroups; a.L = d->ring_len;
    a.num_slots = d->num_slots; a.act_bf16 = d->act_dtype == RSSM_BF16;
    a.out_bf16 = d->out_dtype == RSSM_BF16;
    return m2::dispatch_pn(d->headdim, d->dstate, d->state_dtype, l);
}

extern "C" int rssm_mamba2_decode(const rssm_mamba2_dims* d, void* state, const float* A,
                                  const void* C, const float* D, const void* z, const void* ring_x,
                                  const float* ring_dt, const void* ring_B,
                                  const int32_t* cache_indices, const int32_t* row_wp,
                                  const uint8_t* row_flush, void* workspace, size_t workspace_bytes,
                                  void* y, int32_t* dev_err, rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(A) || !ok_ptr(C) || !ok_ptr(D) || !ok_opt_ptr(z) ||
        !ok_ptr(ring_x) || !ok_ptr(ring_dt) || !ok_ptr(ring_B) || !ok_ptr(cache_indices) ||
        !ok_ptr(row_wp) || !ok_ptr(row_flush) || !ok_ptr(workspace) || !ok_ptr(y))
        return RSSM_ERR_INVALID_ARG;
    rc = rssm_mamba2_precompute(d, A, C, ring_dt, ring_B, cache_indices, row_wp, workspace,
                                workspace_bytes, dev_err, stream);
    if (rc) return rc;
    return rssm_mamba2_output(d, state, C, D, z, ring_x, ring_B, cache_indices, row_wp, row_flush,
                              workspace, workspace_bytes, y, dev_err, stream);
}

extern "C" int rssm_mamba2_full_state_update(const rssm_mamba2_dims* d, void* state, const void* x,
                                             const float* dt_raw, const float* dt_bias,
                                             int dt_softplus, const float* A, const void* B,
                                             const void* C, const float* D, const void* z,
                                             const int32_t* cache_indices, void* y,
                                             int32_t* dev_err, rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(x) || !ok_ptr(dt_raw) || !ok_opt_ptr(dt_bias) || !ok_ptr(A) ||
        !ok_ptr(B) || !ok_ptr(C) || !ok_ptr(D) || !ok_opt_ptr(z) || !ok_ptr(cache_indices) ||
        !ok_ptr(y))
        return RSSM_ERR_INVALID_ARG;
    m2::FullLaunch l{};
    l.stream = (cudaStream_t)stream;
    m2::FullArgs& a = l.a;
    a.state = state; a.x = x; a.dt_raw = dt_raw; a.dt_bias = dt_bias; a.A = A; a.B = B; a.C = C;
    a.D = D; a.z = z; a.ci = cache_indices; a.y = y; a.dev_err = dev_err;
    a.batch = d->batch; a.H = d->nheads; a.G = d->ngroups; a.num_slots = d->num_slots;
    a.act_bf16 = d->act_dtype == RSSM_BF16; a.out_bf16 = d->out_dtype == RSSM_BF16;
    a.softplus = dt_softplus != 0;
    return m2::dispatch_pn(d->headdim, d->dstate, d->state_dtype, l);
}
