// mamba2_small.cu -- the whole Mamba2 ReplaySSM decode step in one launch, for
// small batches.
//
// Pages followed: [M2] "ReplaySSM: cache SSM inputs for faster Mamba2 standard
// decode" (vLLM PR 48018 report): 实现拆解 items 1-3 (precompute, output kernel
// branching per row on is_flush, ring append, per-row write_pos / is_flush), and
// 风险与影响 item 3 (at batch 1-8 the method is launch-bound: a slight slowdown).
//
// At a few rows the two-launch step (per-row prologue, then the streaming output
// kernel) is bound by launch latency, not by bytes. Here one CTA per (row, head)
// does the row's work for its head in one kernel:
//   1. one thread reads the slot's cursor w and the flush decision and issues the
//      bulk copies of the head's checkpoint tile, the ring's x entries 0..w-1 of the
//      head, the B entries 0..w-1 of its group, C and z, while the other threads
//      append this step's x (and, for the first head of a group, B) and dt to the
//      ring at entry w and stage them;
//   3. the head's table -- B_i . C_t, the decay products and coefficients, the
//      checkpoint's decay -- from the staged entries;
//   4. y from the tile and the table (16 lanes per row, reduce-scatters), and on a
//      flush row the fold of entries 0..w into the tile, stored to the pool.
// Right after reading the cursor each CTA counts itself in the row's counter; the
// last CTA of the row to count (every one has read the cursor by then) advances the
// slot's cursor and sets the counter back to 0.
#include "common.cuh"
#include "cursor.cuh"
#include "internal.h"
#include "mamba2.cuh"

namespace rssm {
namespace m2s {

constexpr int kWarps = 2;
constexpr int kThreads = 32 * kWarps;

struct Args {
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
    const uint8_t* force;
    int32_t* slot_wp;
    int32_t* row_wp;
    uint8_t* row_flush;
    void* ring_x;
    float* ring_dt;
    void* ring_B;
    unsigned int* row_count;  // [batch], zero between launches
    void* y;
    int32_t* dev_err;
    int H, G, L, num_slots, act_bf16, out_bf16, softplus;
};

// Shared memory (byte offsets, 16-byte aligned): the tile, x entries [L][P], B entries
// [L][N], C [N], z [P] (activation type), dt [L], table coef [L], a [L], Pm1, B . C [L].
struct Layout {
    int x, B, C, z, dt, tbl, total;
    __host__ __device__ Layout(int P, int N, int SS, int L, int sa) {
        auto up = [](int v) { return (v + 15) & ~15; };
        x = P * N * SS;
        B = x + up(L * P * sa);
        C = B + up(L * N * sa);
        z = C + up(N * sa);
        dt = z + up(P * sa);
        tbl = dt + up(L * 4);
        total = tbl + up((3 * L + 1) * 4);
    }
};

template <int P, int N, class ST>
__global__ void __launch_bounds__(kThreads) step_kernel(const Args a) {
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ uint64_t bar;
    __shared__ int sh_w, sh_f;
    constexpr int SS = ST::bytes;
    const int H = a.H, G = a.G, L = a.L;
    const bool bf = a.act_bf16;
    const int sa = bf ? 2 : 4;
    const int b = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
    const int g = h / (H / G);
    const int t = threadIdx.x, lane = t & 31, wi = t >> 5;
    const Layout lo(P, N, SS, L, sa);
    const int s = a.ci[b];

    // 1. cursor, then the copies of the head's tile and the ring entries before this step
    if (t == 0) {
        int w = -1, f = 0;
        if (s >= a.num_slots) {
            set_dev_err(a.dev_err, RSSM_DEVERR_SLOT);
        } else if (s >= 0) {
            w = a.slot_wp[s];
            if (w < 0 || w >= L) {
                set_dev_err(a.dev_err, RSSM_DEVERR_CURSOR);
                w = -1;
            } else {
                f = (w == L - 1) || (a.force != nullptr && a.force[b] != 0);
            }
        }
        if (h == 0) {
            a.row_wp[b] = w < 0 ? 0 : w;
            a.row_flush[b] = static_cast<uint8_t>(w < 0 ? 0 : f);
        }
        if (w >= 0) {
            // count this CTA in the row's counter; the last of the row's H CTAs to count
            // (every one has read the cursor by then) advances the slot's cursor and sets
            // the counter back to 0
            __threadfence();
            if (atomicAdd(&a.row_count[b], 1u) == (unsigned)H - 1u) {
                __threadfence();
                a.slot_wp[s] = f ? 0 : w + 1;
                atomicExch(&a.row_count[b], 0u);
            }
            mbar_init(&bar, 1);
            fence_barrier_init();
            const uint32_t xb = (uint32_t)w * P * sa, bb = (uint32_t)w * N * sa;
            mbar_arrive_expect_tx(&bar, P * N * SS + xb + bb + N * sa + (a.z ? P * sa : 0));
            bulk_g2s(sm, static_cast<const char*>(a.state) + ((size_t)s * H + h) * P * N * SS,
                     P * N * SS, &bar);
            if (xb)
                bulk_g2s(sm + lo.x, static_cast<const char*>(a.ring_x) + ((size_t)s * H + h) * L * P * sa,
                         xb, &bar);
            if (bb)
                bulk_g2s(sm + lo.B, static_cast<const char*>(a.ring_B) + ((size_t)s * G + g) * L * N * sa,
                         bb, &bar);
            bulk_g2s(sm + lo.C, static_cast<const char*>(a.C) + ((size_t)b * G + g) * N * sa, N * sa, &bar);
            if (a.z)
                bulk_g2s(sm + lo.z, static_cast<const char*>(a.z) + ((size_t)b * H + h) * P * sa, P * sa,
                         &bar);
        }
        sh_w = w;
        sh_f = f;
    }
    __syncthreads();
    const int w = sh_w, f = sh_f;
    if (w < 0) return;  // padding or invalid row: nothing written for it
    // this step's entry: append to the ring and stage it at entry w
    float* dts = reinterpret_cast<float*>(sm + lo.dt);
    {
        const int xc = P * sa / 16;
        const uint4* xs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.x) + ((size_t)b * H + h) * P * sa);
        uint4* xd = reinterpret_cast<uint4*>(static_cast<char*>(a.ring_x) + (((size_t)s * H + h) * L + w) * P * sa);
        for (int c = t; c < xc; c += kThreads) {
            const uint4 v = xs[c];
            xd[c] = v;
            reinterpret_cast<uint4*>(sm + lo.x + (size_t)w * P * sa)[c] = v;
        }
        const int bc = N * sa / 16;
        const uint4* bsrc = reinterpret_cast<const uint4*>(static_cast<const char*>(a.B) + ((size_t)b * G + g) * N * sa);
        uint4* bd = reinterpret_cast<uint4*>(static_cast<char*>(a.ring_B) + (((size_t)s * G + g) * L + w) * N * sa);
        const bool first_of_group = h % (H / G) == 0;
        for (int c = t; c < bc; c += kThreads) {
            const uint4 v = bsrc[c];
            if (first_of_group) bd[c] = v;
            reinterpret_cast<uint4*>(sm + lo.B + (size_t)w * N * sa)[c] = v;
        }
        if (t <= w) {
            float d;
            if (t < w) {
                d = a.ring_dt[((size_t)s * H + h) * L + t];
            } else {
                d = a.dt_raw[(size_t)b * H + h] + (a.dt_bias ? a.dt_bias[h] : 0.f);
                if (a.softplus) d = softplus_f(d);
                a.ring_dt[((size_t)s * H + h) * L + w] = d;
            }
            dts[t] = d;
        }
    }
    if (!mbar_wait_bounded(&bar, 0)) {
        if (t == 0) set_dev_err(a.dev_err, RSSM_DEVERR_TIMEOUT);
        return;
    }
    __syncthreads();

    // 3. the table: bc_i = B_i . C_t (4 threads per entry), then per entry i <= w
    //    P_i = exp(A_h sum_{i<j<=w} dt_j), a_i = P_i dt_i, coef_i = a_i bc_i, and
    //    Pm1 = exp(A_h sum_{j<=w} dt_j)
    float* coef = reinterpret_cast<float*>(sm + lo.tbl);
    float* av = coef + L;
    float* pm1 = av + L;
    float* bcs = pm1 + 1;
    {
        const int i = t >> 2, part = t & 3;
        float acc = 0.f;
        if (i <= w) {
            const uint8_t* Bi = sm + lo.B + (size_t)i * N * sa;
            const uint8_t* Cs = sm + lo.C;
            for (int n = part * 8; n < N; n += 32) {
                float fb[8], fc[8];
                load8(Bi + (size_t)n * sa, bf, fb);
                load8(Cs + (size_t)n * sa, bf, fc);
#pragma unroll
                for (int u = 0; u < 8; ++u) acc = fmaf(fb[u], fc[u], acc);
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        if (part == 0 && i <= w) bcs[i] = acc;
        // entries beyond 16 (rings longer than the 16 entries one pass covers)
        for (int i2 = i + kThreads / 4; i2 <= w; i2 += kThreads / 4) {
            const uint8_t* Bi = sm + lo.B + (size_t)i2 * N * sa;
            float a2 = 0.f;
            for (int n = part * 8; n < N; n += 32) {
                float fb[8], fc[8];
                load8(Bi + (size_t)n * sa, bf, fb);
                load8(sm + lo.C + (size_t)n * sa, bf, fc);
#pragma unroll
                for (int u = 0; u < 8; ++u) a2 = fmaf(fb[u], fc[u], a2);
            }
            a2 += __shfl_xor_sync(0xffffffffu, a2, 1);
            a2 += __shfl_xor_sync(0xffffffffu, a2, 2);
            if (part == 0) bcs[i2] = a2;
        }
    }
    __syncthreads();
    const float Ah = a.A[h];
    for (int i = t; i <= w; i += kThreads) {
        float suffix = 0.f;
        for (int j = i + 1; j <= w; ++j) suffix += dts[j];
        const float Pi = expf(Ah * suffix);
        av[i] = Pi * dts[i];
        coef[i] = av[i] * bcs[i];
        if (i == 0) *pm1 = expf(Ah * (suffix + dts[0]));
    }
    __syncthreads();

    // 4. y: 16 lanes per row (8 columns each), RPI rows per load
    constexpr int PW = P / kWarps, NQ = N / 8, RPI = 32 / NQ, ITER = PW / RPI, NCH = ITER / NQ;
    static_assert(NCH >= 1 && ITER % NQ == 0, "tile shape");
    const int q = lane % NQ, hr = lane / NQ;
    const int row0 = wi * PW + hr;
    const uint8_t* xr = sm + lo.x;
    const float Pm1 = *pm1;
    float part[ITER];
    {
        float c[8];
        load8(sm + lo.C + q * 8 * sa, bf, c);
#pragma unroll
        for (int it = 0; it < ITER; ++it) {
            const int p = row0 + RPI * it;
            float s8[8];
            load8(sm + ((size_t)p * N + q * 8) * SS, ST::bf16, s8);
            float acc = s8[0] * c[0];
#pragma unroll
            for (int j = 1; j < 8; ++j) acc = fmaf(s8[j], c[j], acc);
            part[it] = acc;
        }
    }
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) reduce_scatter<NQ, NQ>(part + ch * NQ);
    const float Dh = a.D[h];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
        const int p = row0 + RPI * (ch * NQ + q);
        float yv = Pm1 * part[ch * NQ];
        for (int i = 0; i <= w; ++i) yv = fmaf(coef[i], load1(xr, i * P + p, bf), yv);
        yv = fmaf(Dh, load1(xr, w * P + p, bf), yv);
        if (a.z) yv *= silu_fast(load1(sm + lo.z, p, bf));
        store1(a.y, ((size_t)b * H + h) * P + p, a.out_bf16, yv);
    }
    if (!f) return;

    // flush: S = Pm1 S0 + sum_{i<=w} a_i x_i B_i^T, stored rounded to the state dtype
    const uint8_t* br = sm + lo.B;
    const size_t tile_e = ((size_t)s * H + h) * P * N;
    constexpr int RC = ITER < 8 ? ITER : 8;
#pragma unroll 1
    for (int t0 = 0; t0 < ITER; t0 += RC) {
        float2 acc[RC][4];
#pragma unroll
        for (int r = 0; r < RC; ++r) {
            const int p = row0 + RPI * (t0 + r);
            float s8[8];
            load8(sm + ((size_t)p * N + q * 8) * SS, ST::bf16, s8);
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[r][k] = make_float2(Pm1 * s8[2 * k], Pm1 * s8[2 * k + 1]);
        }
        for (int i = 0; i <= w; ++i) {
            float bi[8];
            load8(br + ((size_t)i * N + q * 8) * sa, bf, bi);
            const float2 b2[4] = {make_float2(bi[0], bi[1]), make_float2(bi[2], bi[3]),
                                  make_float2(bi[4], bi[5]), make_float2(bi[6], bi[7])};
            const float ai = av[i];
#pragma unroll
            for (int r = 0; r < RC; ++r) {
                const int p = row0 + RPI * (t0 + r);
                const float ax = ai * load1(xr, i * P + p, bf);
                const float2 ax2 = make_float2(ax, ax);
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[r][k] = __ffma2_rn(ax2, b2[k], acc[r][k]);
            }
        }
#pragma unroll
        for (int r = 0; r < RC; ++r) {
            const int p = row0 + RPI * (t0 + r);
            store8(static_cast<char*>(a.state) + (tile_e + (size_t)p * N + q * 8) * SS, ST::bf16,
                   reinterpret_cast<const float*>(acc[r]));
        }
    }
}

}  // namespace m2s

// The one-launch step for `d` (batch <= kSmallStepMaxBatch, round-to-nearest state
// stores, cursor advanced here); RSSM_ERR_UNSUPPORTED when the shape has no
// instance, so the caller takes the two-launch step.
int m2_step_small(const rssm_mamba2_dims* d, const uint8_t* force_flush, int32_t* slot_wp,
                  int32_t* row_wp, uint8_t* row_flush, void* state, const void* x,
                  const float* dt_raw, const float* dt_bias, int dt_softplus, const float* A,
                  const void* B, const void* C, const float* D, const void* z,
                  const int32_t* cache_indices, void* ring_x, float* ring_dt, void* ring_B,
                  void* workspace, void* y, int32_t* dev_err, cudaStream_t stream) {
    m2s::Args a{};
    a.state = state; a.x = x; a.dt_raw = dt_raw; a.dt_bias = dt_bias; a.A = A; a.B = B; a.C = C;
    a.D = D; a.z = z; a.ci = cache_indices; a.force = force_flush; a.slot_wp = slot_wp;
    a.row_wp = row_wp; a.row_flush = row_flush; a.ring_x = ring_x; a.ring_dt = ring_dt;
    a.ring_B = ring_B; a.y = y; a.dev_err = dev_err;
    a.row_count = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) +
                                                  m2::sched_offset(d->batch, d->nheads, d->ring_len)) +
                  m2::kRowCountWord;
    a.H = d->nheads; a.G = d->ngroups; a.L = d->ring_len; a.num_slots = d->num_slots;
    a.act_bf16 = d->act_dtype == RSSM_BF16; a.out_bf16 = d->out_dtype == RSSM_BF16;
    a.softplus = dt_softplus != 0;
    const int sa = a.act_bf16 ? 2 : 4;
    const int SS = d->state_dtype == RSSM_BF16 ? 2 : 4;
    const m2s::Layout lo(d->headdim, d->dstate, SS, d->ring_len, sa);
    const unsigned grid = (unsigned)d->batch * d->nheads;
    auto go = [&](const void* fn, auto launch) -> int {
        if (!ensure_smem_limit(fn, lo.total)) return RSSM_ERR_CUDA;
        launch();
        return launch_status();
    };
#define RSSM_M2S_CASE(PP, NN, STT)                                                                \
    if (d->headdim == PP && d->dstate == NN && SS == STT::bytes)                                  \
        return go(reinterpret_cast<const void*>(m2s::step_kernel<PP, NN, STT>), [&]() {          \
            m2s::step_kernel<PP, NN, STT><<<grid, m2s::kThreads, lo.total, stream>>>(a);        \
        });
    RSSM_M2S_CASE(64, 128, StBF16)
    RSSM_M2S_CASE(64, 128, StF32)
    RSSM_M2S_CASE(128, 128, StBF16)
    RSSM_M2S_CASE(128, 128, StF32)
    RSSM_M2S_CASE(64, 64, StBF16)
    RSSM_M2S_CASE(64, 64, StF32)
    RSSM_M2S_CASE(128, 64, StBF16)
    RSSM_M2S_CASE(128, 64, StF32)
#undef RSSM_M2S_CASE
    return RSSM_ERR_UNSUPPORTED;
}

}  // namespace rssm
