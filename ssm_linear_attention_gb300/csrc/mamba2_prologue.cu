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
//   precompute_kernel   stages C_t, A and the slot's whole dt and B rings in shared
//                       memory with 1-D bulk copies on one mbarrier, then B_i . C_t
//                       per group and the decay suffix products per head (a
//                       segmented warp scan), written as per-(row, head) tables.
//   prepare_kernel      cursor step + ring append + tables: the staging copies are
//                       issued before the cursor is read and the step's inputs are
//                       loaded into registers meanwhile; entry w of the staged
//                       rings is patched from the inputs.
// The prologue is latency-bound work on a few tens of KB per row, so each CTA
// waits for one round trip to memory, not one per loop iteration.
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
    float* ws;             // [batch][H][TBL], then the output kernel's work counter
    unsigned int* sched;   // that counter (zeroed by block 0 of a table-building launch)
};

constexpr int kRowThreads = 256;
constexpr int kRowBlocksPerSM = 4;  // one wave for a batch of up to 4 x SMs rows

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

// Shared memory of the table-building kernels (byte offsets, 16-byte aligned):
// C_t [G][N] and the slot's B ring [G][L][N] in the activation type, A [H], the
// slot's dt ring [H][L] and B . C [G][L] in fp32.
struct ProLayout {
    int c, A, dt, bc, B, total;
    __host__ __device__ ProLayout(int H, int N, int G, int L, int sa) {
        auto up = [](int x) { return (x + 15) & ~15; };
        c = 0;
        A = up(G * N * sa);
        dt = A + up(H * 4);
        bc = dt + up(H * L * 4);
        B = bc + up(G * L * 4);
        total = B + G * L * N * sa;
    }
};

// Stage row b's C_t, A and slot s's whole dt and B rings with 1-D bulk copies
// completing on `bar` (issued by one thread; the dt ring and A fall back to plain
// loads by that thread when their sizes are not multiples of 16 bytes). Returns the
// bytes the barrier expects.
__device__ void stage_issue(const RowArgs& a, int b, int s, uint8_t* sm, uint64_t* bar) {
    const int H = a.H, N = a.N, G = a.G, L = a.L;
    const int sa = a.act_bf16 ? 2 : 4;
    const ProLayout lo(H, N, G, L, sa);
    const bool bulk_dt = ((H * L) & 3) == 0 && (H & 3) == 0;
    uint32_t bytes = G * N * sa + G * L * N * sa + (bulk_dt ? (H + H * L) * 4 : 0);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(sm + lo.c, static_cast<const char*>(a.C) + (size_t)b * G * N * sa, G * N * sa, bar);
    bulk_g2s(sm + lo.B, static_cast<const char*>(a.ring_B) + (size_t)s * G * L * N * sa,
             G * L * N * sa, bar);
    if (bulk_dt) {
        bulk_g2s(sm + lo.A, a.A, H * 4, bar);
        bulk_g2s(sm + lo.dt, a.ring_dt + (size_t)s * H * L, H * L * 4, bar);
    } else {
        float* As = reinterpret_cast<float*>(sm + lo.A);
        float* dts = reinterpret_cast<float*>(sm + lo.dt);
        for (int h = 0; h < H; ++h) As[h] = a.A[h];
        for (int i = 0; i < H * L; ++i) dts[i] = a.ring_dt[(size_t)s * H * L + i];
    }
}

// Row b's tables from the staged rings (entries 0..w):
//   P_i = exp(A_h sum_{i<j<=w} dt_j), coef_i = P_i dt_i (B_i . C_t), a_i = P_i dt_i,
//   Pm1 = exp(A_h sum_{j<=w} dt_j), written straight to the workspace.
// B . C: eight lanes per entry (N/8 dstate columns each, three shuffle levels).
// Tables: a segment of LS = pow2ceil(L) <= 32 lanes per head, lane i = entry i; the
// suffix sums come from a segmented warp scan, so every entry's exp runs in
// parallel and a head's table row is written by consecutive lanes.
__device__ void tables_from_smem(const RowArgs& a, int b, int w, uint8_t* sm) {
    const int H = a.H, N = a.N, G = a.G, L = a.L;
    const int TBL = tbl_floats(L);
    const bool bf = a.act_bf16;
    const int sa = bf ? 2 : 4;
    const int hpg = H / G;
    const ProLayout lo(H, N, G, L, sa);
    const char* craw = reinterpret_cast<const char*>(sm + lo.c);
    const char* braw = reinterpret_cast<const char*>(sm + lo.B);
    const float* As = reinterpret_cast<const float*>(sm + lo.A);
    const float* dts = reinterpret_cast<const float*>(sm + lo.dt);
    float* bc = reinterpret_cast<float*>(sm + lo.bc);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;

    {  // bc[g][i] = B_i . C_t
        const int sub = lane >> 3, part = lane & 7;  // 4 entries per warp, 8 lanes each
        const int per = N / 8;                        // columns per lane
        for (int p0 = warp * 4; p0 < G * (w + 1); p0 += nwarps * 4) {
            const int pair = p0 + sub;
            float acc = 0.f;
            int g = 0, i = 0;
            if (pair < G * (w + 1)) {
                g = pair / (w + 1);
                i = pair - g * (w + 1);
                const char* Bi = braw + ((size_t)g * L + i) * N * sa;
                const char* Cg = craw + (size_t)g * N * sa;
                for (int n = part * per; n < (part + 1) * per; n += 8) {
                    float fb[8], fc[8];
                    load8(Bi + (size_t)n * sa, bf, fb);
                    load8(Cg + (size_t)n * sa, bf, fc);
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc = fmaf(fb[u], fc[u], acc);
                }
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            if (part == 0 && pair < G * (w + 1)) bc[g * L + i] = acc;
        }
    }
    __syncthreads();

    if (L <= 32) {
        int LS = 1;
        while (LS < L) LS <<= 1;
        const int hpw = 32 / LS;  // heads per warp pass
        const int i = lane & (LS - 1);
        for (int h0 = warp * hpw; h0 < H; h0 += nwarps * hpw) {
            const int h = h0 + lane / LS;
            const bool live = h < H;
            const float dti = (live && i <= w) ? dts[h * L + i] : 0.f;
            float incl = dti;  // sum_{i<=j<=w} dt_j after the scan
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                if (off < LS) {
                    const float v = __shfl_down_sync(0xffffffffu, incl, off, LS);
                    if (i + off < LS) incl += v;
                }
            }
            const float total = __shfl_sync(0xffffffffu, incl, 0, LS);
            if (live) {
                const float Ah = As[h];
                float* t = a.ws + ((size_t)b * H + h) * TBL;
                if (i < L) {
                    float ci = 0.f, ai = 0.f;
                    if (i <= w) {
                        const float Pi = expf(Ah * (incl - dti));
                        ai = Pi * dti;
                        ci = ai * bc[(h / hpg) * L + i];
                    }
                    t[i] = ci;
                    t[L + i] = ai;
                }
                for (int e = 2 * L + i; e < TBL; e += LS) t[e] = e == 2 * L ? expf(Ah * total) : 0.f;
            }
        }
    } else {
        for (int h = threadIdx.x; h < H; h += blockDim.x) {
            const int g = h / hpg;
            const float* dh = dts + h * L;
            float* t = a.ws + ((size_t)b * H + h) * TBL;
            const float Ah = As[h];
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

__global__ void __launch_bounds__(kRowThreads, kRowBlocksPerSM) precompute_kernel(const RowArgs a, const int32_t* ci,
                                                                 const int32_t* row_wp,
                                                                 int32_t* dev_err) {
    extern __shared__ __align__(128) uint8_t psm[];
    __shared__ uint64_t bar;
    const int b = blockIdx.x;
    if (b == 0 && threadIdx.x < 2) a.sched[threadIdx.x] = 0u;  // the output kernel's counter
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
// Thread 0 issues the staging copies before it reads the cursor; meanwhile every
// thread loads its share of the step's x, dt and B into registers. After the
// append, entry w of the staged rings is patched with the step's dt and B.
constexpr int kMaxXChunks = 4;  // 16-byte chunks of x held in registers per thread

__global__ void __launch_bounds__(kRowThreads, kRowBlocksPerSM) prepare_kernel(const RowArgs a, const int32_t* ci,
                                                              int advance, const uint8_t* force,
                                                              int32_t* slot_wp, int32_t* row_wp,
                                                              uint8_t* row_flush, int32_t* dev_err) {
    extern __shared__ __align__(128) uint8_t psm[];
    __shared__ uint64_t bar;
    __shared__ int sh_w;
    const int H = a.H, P = a.P, N = a.N, G = a.G, L = a.L;
    const int sa = a.act_bf16 ? 2 : 4;
    const int b = blockIdx.x;
    if (b == 0 && threadIdx.x < 2) a.sched[threadIdx.x] = 0u;  // the output kernel's counter
    const int s = ci[b];
    const bool staged = s >= 0 && s < a.num_slots;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        if (staged) stage_issue(a, b, s, psm, &bar);
        sh_w = advance ? standard_cursor(b, s, a.num_slots, L, slot_wp, force, row_wp, row_flush,
                                         dev_err)
                       : given_cursor(b, s, a.num_slots, L, row_wp, dev_err);
    }
    // the step's inputs, independent of the cursor
    const int xc = P * sa / 16, nx = H * xc;
    const uint4* xs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.x) + (size_t)b * H * P * sa);
    uint4 xr[kMaxXChunks];
#pragma unroll
    for (int u = 0; u < kMaxXChunks; ++u) {
        const int c = threadIdx.x + u * blockDim.x;
        if (c < nx) xr[u] = xs[c];
    }
    const int bcn = N * sa / 16;
    uint4 br = make_uint4(0, 0, 0, 0);
    if (threadIdx.x < G * bcn)
        br = reinterpret_cast<const uint4*>(static_cast<const char*>(a.B) + (size_t)b * G * N * sa)[threadIdx.x];
    float dtr = 0.f;
    if (threadIdx.x < H) dtr = step_dt(a, b, threadIdx.x);
    __syncthreads();
    const int w = sh_w;
    if (staged && !mbar_wait_bounded(&bar, 0)) {
        if (threadIdx.x == 0) set_dev_err(dev_err, RSSM_DEVERR_TIMEOUT);
        return;
    }
    if (w < 0) return;
    // append, from registers, and patch entry w of the staged rings
    const ProLayout lo(H, N, G, L, sa);
#pragma unroll
    for (int u = 0; u < kMaxXChunks; ++u) {
        const int c = threadIdx.x + u * blockDim.x;
        if (c < nx) {
            const int h = c / xc, j = c - (c / xc) * xc;
            reinterpret_cast<uint4*>(static_cast<char*>(a.ring_x) + (((size_t)s * H + h) * L + w) * P * sa)[j] =
                xr[u];
        }
    }
    for (int c = threadIdx.x + kMaxXChunks * blockDim.x; c < nx; c += blockDim.x) {  // wide rows
        const int h = c / xc, j = c - (c / xc) * xc;
        reinterpret_cast<uint4*>(static_cast<char*>(a.ring_x) + (((size_t)s * H + h) * L + w) * P * sa)[j] =
            xs[c];
    }
    float* dts = reinterpret_cast<float*>(psm + lo.dt);
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const float v = h == threadIdx.x ? dtr : step_dt(a, b, h);
        a.ring_dt[((size_t)s * H + h) * L + w] = v;
        dts[h * L + w] = v;
    }
    for (int c = threadIdx.x; c < G * bcn; c += blockDim.x) {
        const uint4 v = c == threadIdx.x ? br
            : reinterpret_cast<const uint4*>(static_cast<const char*>(a.B) + (size_t)b * G * N * sa)[c];
        const int g = c / bcn, j = c - (c / bcn) * bcn;
        reinterpret_cast<uint4*>(static_cast<char*>(a.ring_B) + (((size_t)s * G + g) * L + w) * N * sa)[j] = v;
        reinterpret_cast<uint4*>(psm + lo.B + ((size_t)g * L + w) * N * sa)[j] = v;
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
    return m2::sched_offset(d->batch, d->nheads, d->ring_len) + m2::kSchedBytes;
}

// Shared-memory size of the table-building kernels, checked and opted in.
static int m2_prologue_smem(const rssm_mamba2_dims* d, const void* kernel, int* smem) {
    *smem = m2::ProLayout(d->nheads, d->dstate, d->ngroups, d->ring_len,
                          d->act_dtype == RSSM_BF16 ? 2 : 4).total;
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
    ra.sched = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) +
                                               m2::sched_offset(d->batch, d->nheads, d->ring_len));
    m2::precompute_kernel<<<d->batch, m2::kRowThreads, smem, (cudaStream_t)stream>>>(ra, cache_indices, row_wp,
                                                                                      dev_err);
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
    ra.sched = reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) +
                                               m2::sched_offset(d->batch, d->nheads, d->ring_len));
    rc = m2_prologue_smem(d, reinterpret_cast<const void*>(m2::prepare_kernel), &smem);
    if (rc) return rc;
    m2::prepare_kernel<<<d->batch, m2::kRowThreads, smem, (cudaStream_t)stream>>>(
        ra, cache_indices, advance ? 1 : 0, force_flush, slot_wp, row_wp, row_flush, dev_err);
    return launch_status();
}
