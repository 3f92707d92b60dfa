// mamba2_spec.cu -- speculative verify for Mamba2 on the circular ReplaySSM ring.
//
// Pages followed: "ReplaySSM: cache SSM inputs for faster Mamba2 standard decode",
// 关联脉络 (the full design, PR 47576, covers Mamba2 and GDN with standard and
// speculative decode); "[GDN] Support ReplaySSM Ring Spec-Verify", 实现拆解 items
// 2-4 (circular ring with cursors write_pos / cache_base / is_flush, per-draft
// outputs from checkpoint + ring without per-draft states, a fold of the committed
// entries into the checkpoint before a round that would overrun the ring, a commit
// that only moves cursors), read for Mamba2.
//
// Cursors per slot: cnt (committed, unfolded entries), base (oldest entry's ring
// position), flush (fold pending). A round with history c = cnt entries at
// positions (base + i) % L scores T drafts; draft j's entry goes to position
// (base + c + j) % L. With m = c + j and entries i = 0..m (history, then drafts),
// the recurrence h <- dA h + dt x B^T, y = h C + D x unrolls to
//   y_j = (prod_{i<=m} dA_i) S0 C_j + sum_{i<=m} (prod_{l=i+1..m} dA_l) dt_i (B_i . C_j) x_i
//         + D x_j,   gated by silu(z_j),
// so each draft needs its own decay and B.C_j table but S0 is read once for all.
// A pending fold is the Mamba2 flush over the committed entries:
//   S0 <- (prod_{i<cnt} dA_i) S0 + sum_{i<cnt} (prod_{l=i+1..cnt-1} dA_l) dt_i x_i B_i^T.
//
// Two launches: a prologue whose CTAs either fold one (row, head) tile of a slot
// with a pending fold or build one row's tables; then the verify (warp-specialised
// pipeline over (row, head) tiles), which also appends the drafts to the ring.
// The commit is rssm_advance_cursors(RSSM_CURSOR_SPEC_COMMIT).
#include "common.cuh"
#include "internal.h"
#include "mamba2.cuh"
#include "pipeline.cuh"

namespace rssm {
namespace m2spec {

constexpr int kMaxT = 4;
constexpr int kThreads = 128;  // prologue CTA

// Per-(row, head) table: coef[T][L] (draft j's coefficient of entry i), Pm1[T],
// the drafts' dt[T], padded to 4 floats.
__host__ __device__ inline int tbl_floats(int L, int T) { return (T * L + 2 * T + 3) & ~3; }

// Effective history at verify time (count, oldest position); false when the cursors
// are outside the ring or the drafts would not fit.
__device__ __forceinline__ bool history(int cnt, int base, int flush, int L, int T, int* c,
                                        int* base_eff) {
    if (cnt < 0 || cnt > L || base < 0 || base >= L) return false;
    *c = flush ? 0 : cnt;
    *base_eff = flush ? (base + cnt) % L : base;
    return *c + T <= L;
}

struct ProArgs {
    void* state;
    const float* dt_raw;
    const float* dt_bias;
    const float* A;
    const void* B;
    const void* C;
    const void* ring_x;
    const float* ring_dt;
    const void* ring_B;
    const int32_t* ci;
    const int32_t* slot_cnt;
    const int32_t* slot_base;
    const uint8_t* slot_flush;
    float* ws;
    int32_t* dev_err;
    int batch, T, H, P, N, G, L, num_slots, act_bf16, state_bf16, softplus;
    int n_tbl;   // table CTAs (batch * G), after the fold CTAs
    int n_fold;  // persistent fold CTAs, first in the grid
};

__device__ __forceinline__ float ring_dt_at(const ProArgs& a, int s, int h, int pos) {
    return a.ring_dt[((size_t)s * a.H + h) * a.L + pos];
}

// Fold of one (row, head) tile of a slot whose fold is pending:
//   S0 <- Pm1 S0 + sum_{i<cnt} a_i x_i B_i^T,  a_i = exp(A sum_{l>i} dt_l) dt_i.
// Thread t owns 4 consecutive dstate columns (n0 = 4 (t mod N/4)) of RPT consecutive
// headdim rows (RPT = P N / 512: 8, 16 or 32, a multiple of 4). One round trip: the
// committed x and B entries are copied into shared memory asynchronously (no
// registers) while the thread's state rows (up to 16 of them; a float32 state: 8)
// and the entries' dt are loaded into registers. A short pass then turns the staged
// entries into float32 (x scaled by a_i), and the update runs 4 rows per pass as
// packed two-wide FMAs. SBF / ABF: the state / the activations are bf16.
template <bool BF>
struct Raw4 {  // 4 state elements as loaded: bf16 pairs or float32
    uint2 u;
    __device__ __forceinline__ void load(const void* base, long i) {
        u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + i);
    }
    __device__ __forceinline__ float4 f() const {
        return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
    }
};
template <>
struct Raw4<false> {
    float4 v;
    __device__ __forceinline__ void load(const void* base, long i) {
        v = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    }
    __device__ __forceinline__ float4 f() const { return v; }
};

// Shared memory of the fold role (floats): x [L][P] and B [L][N] in float32, a_i and
// Pm1 [L + 1] (padded to 4), then the raw staged entries (activation dtype).
__host__ __device__ inline int fold_smem_floats(int P, int N, int L) {
    return L * P + L * N + ((L + 1 + 3) & ~3) + L * (P + N);
}

template <bool SBF, bool ABF>
__device__ void fold_tile(const ProArgs& a, int b, int h, float* sm) {
    const int s = a.ci[b];
    const int cnt = a.slot_cnt[s], base = a.slot_base[s], L = a.L;
    if (cnt <= 0 || cnt > L || base < 0 || base >= L) return;
    const int P = a.P, N = a.N, g = h / (a.H / a.G);
    constexpr int ss = SBF ? 2 : 4, sa = ABF ? 2 : 4;
    const int t = threadIdx.x;
    float* xs = sm;                                  // [cnt][P]: a_i x_i[p]
    float* bs = xs + L * P;                          // [cnt][N]
    float* cf = bs + L * N;                          // [cnt] a_i, then Pm1
    uint8_t* xr = reinterpret_cast<uint8_t*>(cf + ((L + 1 + 3) & ~3));  // [cnt][P] raw
    uint8_t* br = xr + (size_t)L * P * sa;                             // [cnt][N] raw
    const int ncg = N / 4;
    const int n0 = (t % ncg) * 4, rg = t / ncg;
    const int RPT = P * ncg / kThreads;
    const int p0 = rg * RPT;
    char* st = static_cast<char*>(a.state) + ((size_t)s * a.H + h) * P * N * ss;
    constexpr int RB = 4;               // rows per pass (few live accumulators)
    constexpr int RMAX = SBF ? 16 : 8;  // rows loaded per round trip, held in registers
    const int rl = RPT < RMAX ? RPT : RMAX;

    __syncthreads();  // the previous tile's readers are done with the buffers
    {
        const int xc = P * sa / 16, bc_ = N * sa / 16;  // 16-byte chunks per entry
        const char* xsrc = static_cast<const char*>(a.ring_x) + ((size_t)s * a.H + h) * L * P * sa;
        const char* bsrc = static_cast<const char*>(a.ring_B) + ((size_t)s * a.G + g) * L * N * sa;
        for (int e = t; e < cnt * (xc + bc_); e += kThreads) {
            if (e < cnt * xc) {
                const int i = e / xc, c16 = e - i * xc;
                cp_async16(xr + (size_t)e * 16, xsrc + (size_t)((base + i) % L) * P * sa + c16 * 16);
            } else {
                const int e2 = e - cnt * xc, i = e2 / bc_, c16 = e2 - i * bc_;
                cp_async16(br + (size_t)e2 * 16, bsrc + (size_t)((base + i) % L) * N * sa + c16 * 16);
            }
        }
        cp_async_commit();
    }
    Raw4<SBF> sv[RMAX];
#pragma unroll
    for (int k = 0; k < RMAX; ++k)
        if (k < rl) sv[k].load(st, (long)(p0 + k) * N + n0);
    const float dti = t < cnt ? ring_dt_at(a, s, h, (base + t) % L) : 0.f;
    if (t < 32) {
        // a_i = prod_{l>i} dA_l * dt_i from a suffix sum over the committed entries
        const float Ah = a.A[h];
        float suf = dti;  // inclusive suffix sum: sum_{l>=t} dt_l
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_down_sync(kFull, suf, o);
            if (t + o < 32) suf += v;
        }
        if (t < cnt) cf[t] = expf(Ah * (suf - dti)) * dti;
        const float total = __shfl_sync(kFull, suf, 0);
        if (t == 0) cf[cnt] = expf(Ah * total);
    }
    cp_async_wait_all();
    __syncthreads();
    // the staged entries in float32, x scaled by a_i (4 elements at a time)
    for (int e = t; e < cnt * (P + N) / 4; e += kThreads) {
        float f[4];
        if (e < cnt * P / 4) {
            load4(xr, e * 4, ABF, f);
            const float c_ = cf[e / (P / 4)];
            *reinterpret_cast<float4*>(xs + e * 4) = make_float4(c_ * f[0], c_ * f[1], c_ * f[2], c_ * f[3]);
        } else {
            const int e2 = e - cnt * P / 4;
            load4(br, e2 * 4, ABF, f);
            *reinterpret_cast<float4*>(bs + e2 * 4) = make_float4(f[0], f[1], f[2], f[3]);
        }
    }
    __syncthreads();
    const float Pm1 = cf[cnt];
    for (int r0 = 0; r0 < RPT; r0 += RMAX) {
        if (r0 > 0) {  // only when the thread has more rows than one round holds
#pragma unroll
            for (int k = 0; k < RMAX; ++k)
                if (r0 + k < RPT) sv[k].load(st, (long)(p0 + r0 + k) * N + n0);
        }
#pragma unroll
        for (int q = 0; q < RMAX; q += RB) {
            if (r0 + q >= RPT) break;
            float2 acc[RB][2];
#pragma unroll
            for (int k = 0; k < RB; ++k) {
                const float4 f = sv[q + k].f();
                acc[k][0] = make_float2(Pm1 * f.x, Pm1 * f.y);
                acc[k][1] = make_float2(Pm1 * f.z, Pm1 * f.w);
            }
            const int pr = p0 + r0 + q;  // first row of this pass
            for (int i = 0; i < cnt; ++i) {
                const float4 b4 = *reinterpret_cast<const float4*>(bs + i * N + n0);
                const float4 x4 = *reinterpret_cast<const float4*>(xs + i * P + pr);
                const float2 blo = make_float2(b4.x, b4.y), bhi = make_float2(b4.z, b4.w);
                const float xk[RB] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
                for (int k = 0; k < RB; ++k) {
                    const float2 x2 = make_float2(xk[k], xk[k]);
                    acc[k][0] = __ffma2_rn(x2, blo, acc[k][0]);
                    acc[k][1] = __ffma2_rn(x2, bhi, acc[k][1]);
                }
            }
#pragma unroll
            for (int k = 0; k < RB; ++k) {
                char* d = st + (size_t)((pr + k) * N + n0) * ss;
                if constexpr (SBF) {
                    *reinterpret_cast<uint2*>(d) = make_uint2(pack_bf16x2(acc[k][0].x, acc[k][0].y),
                                                              pack_bf16x2(acc[k][1].x, acc[k][1].y));
                } else {
                    *reinterpret_cast<float4*>(d) =
                        make_float4(acc[k][0].x, acc[k][0].y, acc[k][1].x, acc[k][1].y);
                }
            }
        }
    }
}

// Fold role (CTA f of n_fold): every fold CTA builds the same ascending list of the
// rows with a pending fold (ballots over the batch), and the list's (row, head)
// tiles are dealt round-robin over the fold CTAs. Rows beyond kFoldRows are
// checked per tile instead.
constexpr int kFoldRows = 1024;

template <bool SBF, bool ABF>
__device__ void fold_role(const ProArgs& a, int f, float* sm) {
    __shared__ int rows[kFoldRows];
    __shared__ int wsum[kThreads / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    auto pending = [&](int b) {
        const int s = a.ci[b];
        return s >= 0 && s < a.num_slots && a.slot_flush[s];
    };
    const int nl = a.batch < kFoldRows ? a.batch : kFoldRows;  // rows taken into the list
    int base = 0;
    for (int b0 = 0; b0 < nl; b0 += kThreads) {
        const int b = b0 + t;
        const bool flag = b < nl && pending(b);
        const unsigned m = __ballot_sync(kFull, flag);
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
    const int tiles = base * a.H;
    for (int x = f; x < tiles; x += a.n_fold) {
        const int ri = x / a.H;
        fold_tile<SBF, ABF>(a, rows[ri], x - ri * a.H, sm);
    }
    // rows past the list (batches above kFoldRows): tile by tile
    const long rest = (long)(a.batch - nl) * a.H;
    for (long x = f; x < rest; x += a.n_fold) {
        const int b = nl + (int)(x / a.H);
        if (pending(b)) fold_tile<SBF, ABF>(a, b, (int)(x - (long)(b - nl) * a.H), sm);
    }
}

// Table role: one (row, group). bc[i][j] = B_i . C_j for the row's entries i
// (history from the ring, then the drafts' B) and drafts j; then per (head of the
// group, draft) the decay suffix sums give coef[j][i], Pm1[j], and the drafts' dt.
// Every global load is issued before the first use.
__device__ void group_tables(const ProArgs& a, int b, int g, float* sm) {
    const int s = a.ci[b];
    if (s < 0) return;
    if (s >= a.num_slots) {
        if (threadIdx.x == 0 && g == 0) set_dev_err(a.dev_err, RSSM_DEVERR_SLOT);
        return;
    }
    const int L = a.L, T = a.T, H = a.H, N = a.N, G = a.G;
    int c, base_eff;
    if (!history(a.slot_cnt[s], a.slot_base[s], a.slot_flush[s], L, T, &c, &base_eff)) {
        if (threadIdx.x == 0 && g == 0) set_dev_err(a.dev_err, RSSM_DEVERR_CURSOR);
        return;
    }
    const int ne = c + T;  // entries: history, then drafts
    const int hpg = H / G;
    const bool bf = a.act_bf16;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    float* Cs = sm;                 // [T][N]
    float* Bs = Cs + kMaxT * N;     // [ne][N]
    float* dts = Bs + L * N;        // [hpg][ne]
    float* bc = dts + hpg * L;      // [ne][T]
    const int nc4 = T * (N / 4), nb4 = ne * (N / 4), nd = hpg * ne;
    constexpr int KC = (kMaxT * 128 / 4 + kThreads - 1) / kThreads;
    constexpr int KB = (32 * 128 / 4 + kThreads - 1) / kThreads;
    float cv[KC][4], bv[KB][4];
#pragma unroll
    for (int u = 0; u < KC; ++u) {
        const int e = t + u * kThreads;
        if (e < nc4) {
            const int j = e / (N / 4), c4 = e - j * (N / 4);
            load4(a.C, (int)((((size_t)b * T + j) * G + g) * N) + c4 * 4, bf, cv[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < KB; ++u) {
        const int e = t + u * kThreads;
        if (e < nb4) {
            const int i = e / (N / 4), c4 = e - i * (N / 4);
            if (i < c)
                load4(a.ring_B, (int)((((size_t)s * G + g) * L + (base_eff + i) % L) * N) + c4 * 4, bf, bv[u]);
            else
                load4(a.B, (int)((((size_t)b * T + (i - c)) * G + g) * N) + c4 * 4, bf, bv[u]);
        }
    }
    for (int e0 = t; e0 < nd; e0 += 4 * kThreads) {  // four loads in flight per thread
        float dv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            if (e < nd) {
                const int hl = e / ne, i = e - (e / ne) * ne, h = g * hpg + hl;
                dv[u] = i < c ? ring_dt_at(a, s, h, (base_eff + i) % L)
                              : a.dt_raw[((size_t)b * T + (i - c)) * H + h] + (a.dt_bias ? a.dt_bias[h] : 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            if (e < nd) {
                const int i = e - (e / ne) * ne;
                dts[e] = (i >= c && a.softplus) ? softplus_f(dv[u]) : dv[u];
            }
        }
    }
#pragma unroll
    for (int u = 0; u < KC; ++u) {
        const int e = t + u * kThreads;
        if (e < nc4) *reinterpret_cast<float4*>(Cs + e * 4) = make_float4(cv[u][0], cv[u][1], cv[u][2], cv[u][3]);
    }
#pragma unroll
    for (int u = 0; u < KB; ++u) {
        const int e = t + u * kThreads;
        if (e < nb4) *reinterpret_cast<float4*>(Bs + e * 4) = make_float4(bv[u][0], bv[u][1], bv[u][2], bv[u][3]);
    }
    __syncthreads();
    // B_i . C_j: a warp per entry i, lanes over dstate (4 columns each), one
    // reduce-scatter over the T dots
    for (int i = warp; i < ne; i += kThreads / 32) {
        float part[kMaxT];
#pragma unroll
        for (int j = 0; j < kMaxT; ++j) part[j] = 0.f;
        for (int n = lane * 4; n < N; n += 128) {
            const float4 b4 = *reinterpret_cast<const float4*>(Bs + i * N + n);
#pragma unroll
            for (int j = 0; j < kMaxT; ++j) {
                if (j < T) {
                    const float4 c4 = *reinterpret_cast<const float4*>(Cs + j * N + n);
                    part[j] = fmaf(b4.x, c4.x, fmaf(b4.y, c4.y, fmaf(b4.z, c4.z, fmaf(b4.w, c4.w, part[j]))));
                }
            }
        }
        const int e = reduce_scatter<kMaxT, 32>(part);
        if ((lane & 7) == 0 && e < T) bc[i * T + e] = part[0];
    }
    __syncthreads();
    const int TB = tbl_floats(L, T);
    for (int e = t; e < hpg * T; e += kThreads) {
        const int hl = e / T, j = e - (e / T) * T, h = g * hpg + hl;
        const int m = c + j;
        const float Ah = a.A[h];
        float* tb = a.ws + ((size_t)b * H + h) * TB;
        const float* dh = dts + hl * ne;
        float cum = 0.f;
        for (int i = m; i >= 0; --i) {
            const float dti = dh[i];
            tb[j * L + i] = expf(Ah * cum) * dti * bc[i * T + j];
            cum += dti;
        }
        tb[T * L + j] = expf(Ah * cum);
        tb[T * L + T + j] = dh[m];
    }
}

// Grid: the persistent fold CTAs (the long ones, they start first and hold part of
// each SM), then the table CTAs (one per (row, group)), which fill the other slots.
// One instance per state / activation dtype pair.
template <bool SBF, bool ABF>
__global__ void __launch_bounds__(kThreads, 6) prologue_kernel(const ProArgs a) {
    extern __shared__ __align__(16) float psm[];
    const int blk = blockIdx.x;
    if (blk < a.n_fold) {
        fold_role<SBF, ABF>(a, blk, psm);
        return;
    }
    const int tb = blk - a.n_fold;
    group_tables(a, tb / a.G, tb - (tb / a.G) * a.G, psm);
}

inline int pro_smem_floats(int H, int P, int N, int G, int L) {
    const int tables = kMaxT * N + L * N + (H / G) * L + L * kMaxT;
    const int fold = fold_smem_floats(P, N, L);
    return tables > fold ? tables : fold;
}

// ----------------------------------------------------------------------------
// verify: one (row, head) tile per item; a consumer group of two warps, each with
// half of the headdim rows; lane = (row group hr, dstate chunk q) as in the decode
// output kernel. The T dot products S0 . C_j per row reduce with reduce-scatters.
// ----------------------------------------------------------------------------

constexpr int kGroupWarps = 2;

template <int P, int N, class ST, int T>
struct VerPolicy {
    static constexpr int kGroup = kGroupWarps;
    static constexpr int SS = ST::bytes;
    static constexpr int TILE = P * N * SS;
    static constexpr int PW = P / kGroupWarps;
    static constexpr int NQ = N / 8;
    static constexpr int RPI = 32 / NQ;
    static constexpr int ITER = PW / RPI;
    static constexpr int NCH = ITER / NQ;
    static_assert(NCH >= 1 && ITER % NQ == 0, "tile shape");
    struct Args {
        const void* state;
        const void* x;
        const float* D;
        const void* z;
        const void* B;
        const void* C;
        void* ring_x;
        float* ring_dt;
        void* ring_B;
        const int32_t* ci;
        const int32_t* slot_cnt;
        const int32_t* slot_base;
        const uint8_t* slot_flush;
        const float* ws;
        void* y;
        int32_t* dev_err;
        int batch, H, G, L, num_slots, act_bf16, out_bf16;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
        int off_xh, off_xd, off_z, off_C, off_B, off_tbl;
    };
    struct Meta {
        int valid, s, b, h, c, base_eff;
    };

    static __device__ int n_items(const Args& a) { return a.batch * a.H; }

    static __device__ int4 prefetch(const Args& a, int item) {
        const int b = item / a.H;
        const int s = a.ci[b];
        int c = 0, be = 0;
        if (s >= 0 && s < a.num_slots) {
            if (!history(a.slot_cnt[s], a.slot_base[s], a.slot_flush[s], a.L, T, &c, &be)) c = -1;
        }
        return make_int4(s, c, be, b);
    }

    static __device__ void issue(const Args& a, int item, int4 r, Meta* meta, uint8_t* sb,
                                 uint64_t* full, uint64_t pol) {
        const int b = r.w, h = item - r.w * a.H;
        Meta m{0, r.x, b, h, r.y, r.z};
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
        const int sa = a.act_bf16 ? 2 : 4;
        const int L = a.L, c = m.c;
        const int g = h / (a.H / a.G);
        const int TB = tbl_floats(L, T);
        const uint32_t xb = P * sa, nb = N * sa;
        const bool wb = h % (a.H / a.G) == 0;  // this tile appends the group's drafts' B
        mbar_arrive_expect_tx(full, TILE + (c + T) * xb + (a.z ? T * xb : 0) + (wb ? 2 : 1) * T * nb +
                                        TB * 4);
        bulk_g2s_hint(sb, static_cast<const char*>(a.state) + ((size_t)m.s * a.H + h) * TILE, TILE,
                      full, pol);
        // history x: ring positions base_eff .. base_eff + c - 1 (at most two runs)
        const char* xr = static_cast<const char*>(a.ring_x) + ((size_t)m.s * a.H + h) * L * xb;
        const int run1 = m.base_eff + c <= L ? c : L - m.base_eff;
        if (run1 > 0) bulk_g2s(sb + a.off_xh, xr + (size_t)m.base_eff * xb, run1 * xb, full);
        if (c > run1) bulk_g2s(sb + a.off_xh + run1 * xb, xr, (c - run1) * xb, full);
#pragma unroll
        for (int j = 0; j < T; ++j) {
            const size_t bj = (size_t)b * T + j;
            bulk_g2s(sb + a.off_xd + j * xb, static_cast<const char*>(a.x) + (bj * a.H + h) * xb, xb,
                     full);
            if (a.z)
                bulk_g2s(sb + a.off_z + j * xb, static_cast<const char*>(a.z) + (bj * a.H + h) * xb,
                         xb, full);
            bulk_g2s(sb + a.off_C + j * nb, static_cast<const char*>(a.C) + (bj * a.G + g) * nb, nb,
                     full);
            if (wb)
                bulk_g2s(sb + a.off_B + j * nb, static_cast<const char*>(a.B) + (bj * a.G + g) * nb,
                         nb, full);
        }
        bulk_g2s(sb + a.off_tbl, a.ws + ((size_t)b * a.H + h) * TB, TB * 4, full);
    }

    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb, uint8_t*,
                                   int lane, int wi) {
        if (!m.valid) return;
        const bool bf = a.act_bf16;
        const int sa = bf ? 2 : 4;
        const int L = a.L, c = m.c;
        const int q = lane % NQ, hr = lane / NQ;
        const int row0 = wi * PW + hr;
        const float* tbl = reinterpret_cast<const float*>(sb + a.off_tbl);
        const uint8_t* xh = sb + a.off_xh;
        const uint8_t* xd = sb + a.off_xd;
        float part[T][ITER];
        if (ST::bf16 && bf) {
            uint4 cpk[T];
#pragma unroll
            for (int j = 0; j < T; ++j)
                cpk[j] = *reinterpret_cast<const uint4*>(sb + a.off_C + j * N * 2 + q * 16);
#pragma unroll
            for (int t = 0; t < ITER; ++t) {
                const int p = row0 + RPI * t;
                const uint4 s8 = *reinterpret_cast<const uint4*>(sb + ((size_t)p * N + q * 8) * SS);
#pragma unroll
                for (int j = 0; j < T; ++j) part[j][t] = dot8_bf16(s8, cpk[j], 0.f);
            }
        } else {
            float cv[T][8];
#pragma unroll
            for (int j = 0; j < T; ++j) load8(sb + a.off_C + (j * N + q * 8) * sa, bf, cv[j]);
#pragma unroll
            for (int t = 0; t < ITER; ++t) {
                const int p = row0 + RPI * t;
                float s8[8];
                load8(sb + ((size_t)p * N + q * 8) * SS, ST::bf16, s8);
#pragma unroll
                for (int j = 0; j < T; ++j) {
                    float acc = s8[0] * cv[j][0];
#pragma unroll
                    for (int e = 1; e < 8; ++e) acc = fmaf(s8[e], cv[j][e], acc);
                    part[j][t] = acc;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < T; ++j)
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) reduce_scatter<NQ, NQ>(part[j] + ch * NQ);
        const float Dh = __ldg(a.D + m.h);
        const int pos0 = m.base_eff + c;
        int posj[T];  // the drafts' ring positions
        {
            int p_ = pos0 >= L ? pos0 - L : pos0;
#pragma unroll
            for (int j = 0; j < T; ++j) {
                posj[j] = p_;
                p_ = p_ + 1 == L ? 0 : p_ + 1;
            }
        }
        const size_t ystep = (size_t)a.H * P;
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            const int p = row0 + RPI * (ch * NQ + q);
            float hist[T];
#pragma unroll
            for (int j = 0; j < T; ++j) hist[j] = 0.f;
            for (int i = 0; i < c; ++i) {
                const float xi = load1(xh, i * P + p, bf);
#pragma unroll
                for (int j = 0; j < T; ++j) hist[j] = fmaf(tbl[j * L + i], xi, hist[j]);
            }
            float xdv[T], yv[T];
#pragma unroll
            for (int j = 0; j < T; ++j) xdv[j] = load1(xd, j * P + p, bf);
#pragma unroll
            for (int j = 0; j < T; ++j) {
                float acc = fmaf(tbl[T * L + j], part[j][ch * NQ], hist[j]);
#pragma unroll
                for (int jj = 0; jj <= j; ++jj) acc = fmaf(tbl[j * L + c + jj], xdv[jj], acc);
                acc = fmaf(Dh, xdv[j], acc);
                if (a.z) acc *= silu_fast(load1(sb + a.off_z, j * P + p, bf));
                yv[j] = acc;
            }
            // the outputs, then the drafts' x into the ring (exact: the value came in
            // this dtype)
            const size_t y0 = (((size_t)m.b * T) * a.H + m.h) * P + p;
            const size_t x0 = ((size_t)m.s * a.H + m.h) * L * P + p;
#pragma unroll
            for (int j = 0; j < T; ++j) {
                store1(a.y, (long)(y0 + j * ystep), a.out_bf16, yv[j]);
                store1(a.ring_x, (long)(x0 + (size_t)posj[j] * P), bf, xdv[j]);
            }
        }
        // the drafts' dt (one lane) and B (first head of each group, warp 0)
        if (wi == 0 && lane < T)
            a.ring_dt[((size_t)m.s * a.H + m.h) * L + (pos0 + lane) % L] = tbl[T * L + T + lane];
        if (wi == 0 && m.h % (a.H / a.G) == 0) {
            // from the stage, 16 bytes per lane and store
            const int g = m.h / (a.H / a.G);
            const int cpr = N * sa / 16;  // 16-byte chunks per entry
            for (int e = lane; e < T * cpr; e += 32) {
                const int j = e / cpr, c16 = e - (e / cpr) * cpr;
                const uint4 v = *reinterpret_cast<const uint4*>(sb + a.off_B + (size_t)e * 16);
                char* dst = static_cast<char*>(a.ring_B) +
                            (((size_t)m.s * a.G + g) * L + (pos0 + j) % L) * N * sa;
                reinterpret_cast<uint4*>(dst)[c16] = v;
            }
        }
    }
};

}  // namespace m2spec
}  // namespace rssm

using namespace rssm;

namespace {

template <int T>
struct VerLaunch {
        const rssm_mamba2_dims* d;
        const void *state, *x, *z, *B, *C;
        const float *D, *ws;
        void *ring_x, *ring_B, *y;
        float* ring_dt;
        const int32_t *ci, *slot_cnt, *slot_base;
        const uint8_t* slot_flush;
        int32_t* dev_err;
        cudaStream_t st;
        template <int PP, int NN, class ST>
        int go() {
            using Pol = m2spec::VerPolicy<PP, NN, ST, T>;
            typename Pol::Args va{};
            va.state = state; va.x = x; va.D = D; va.z = z; va.B = B; va.C = C;
            va.ring_x = ring_x; va.ring_dt = ring_dt; va.ring_B = ring_B; va.ci = ci;
            va.slot_cnt = slot_cnt; va.slot_base = slot_base; va.slot_flush = slot_flush;
            va.ws = ws; va.y = y; va.dev_err = dev_err;
            va.batch = d->batch; va.H = d->nheads; va.G = d->ngroups; va.L = d->ring_len;
            va.num_slots = d->num_slots; va.act_bf16 = d->act_dtype == RSSM_BF16;
            va.out_bf16 = d->out_dtype == RSSM_BF16;
            const int sa = va.act_bf16 ? 2 : 4;
            int off = Pol::TILE;
            va.off_xh = off;  off += (d->ring_len - T) * PP * sa;
            va.off_xd = off;  off += T * PP * sa;
            va.off_z = off;   off += T * PP * sa;
            va.off_C = off;   off += T * NN * sa;
            va.off_B = off;   off += T * NN * sa;
            va.off_tbl = off; off += m2spec::tbl_floats(d->ring_len, T) * 4;
            const int stage_bytes = (off + 127) & ~127;
            return launch_pipe<Pol>(va, stage_bytes, 0, Pol::TILE, (long)d->batch * d->nheads, st);
        }
};

template <int T>
int m2spec_launch(const rssm_mamba2_dims* d, void* state, const void* x, const float* dt_raw,
                  const float* dt_bias, int dt_softplus, const float* A, const void* B,
                  const void* C, const float* D, const void* z, void* ring_x, float* ring_dt,
                  void* ring_B, const int32_t* ci, const int32_t* slot_cnt,
                  const int32_t* slot_base, const uint8_t* slot_flush, void* workspace, void* y,
                  int32_t* dev_err, cudaStream_t st) {
    DeviceInfo di;
    if (!device_info(&di)) return RSSM_ERR_CUDA;
    const int H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups, L = d->ring_len;
    // 1. folds of slots with a pending fold, and the tables
    m2spec::ProArgs pa{};
    pa.state = state; pa.dt_raw = dt_raw; pa.dt_bias = dt_bias; pa.A = A; pa.B = B; pa.C = C;
    pa.ring_x = ring_x; pa.ring_dt = ring_dt; pa.ring_B = ring_B; pa.ci = ci;
    pa.slot_cnt = slot_cnt; pa.slot_base = slot_base; pa.slot_flush = slot_flush;
    pa.ws = static_cast<float*>(workspace); pa.dev_err = dev_err;
    pa.batch = d->batch; pa.T = T; pa.H = H; pa.P = P; pa.N = N; pa.G = G; pa.L = L;
    pa.num_slots = d->num_slots; pa.act_bf16 = d->act_dtype == RSSM_BF16;
    pa.state_bf16 = d->state_dtype == RSSM_BF16; pa.softplus = dt_softplus != 0;
    const int psmem = m2spec::pro_smem_floats(H, P, N, G, L) * 4;
    if (psmem > di.max_smem_optin) return RSSM_ERR_UNSUPPORTED;
    const bool sbf = d->state_dtype == RSSM_BF16, abf = d->act_dtype == RSSM_BF16;
    auto kern = sbf ? (abf ? m2spec::prologue_kernel<true, true> : m2spec::prologue_kernel<true, false>)
                    : (abf ? m2spec::prologue_kernel<false, true> : m2spec::prologue_kernel<false, false>);
    if (psmem > 48 * 1024 && !ensure_smem_limit(reinterpret_cast<const void*>(kern), psmem))
        return RSSM_ERR_CUDA;
    pa.n_tbl = d->batch * G;
    {
        long nf = (long)di.sm_count * 4;  // four of the six CTA slots of an SM
        const long tiles = (long)d->batch * H;
        if (nf > tiles) nf = tiles;
        pa.n_fold = (int)nf;
    }
    const long blocks = (long)pa.n_tbl + pa.n_fold;
    kern<<<(unsigned)blocks, m2spec::kThreads, psmem, st>>>(pa);
    if (launch_status()) return RSSM_ERR_CUDA;

    // 2. verify (and the drafts' ring entries)
    VerLaunch<T> g{d, state, x, z, B, C, D, static_cast<const float*>(workspace), ring_x, ring_B, y, ring_dt,
        ci, slot_cnt, slot_base, slot_flush, dev_err, st};
#define RSSM_M2S_CASE(PP, NN)                                                 \
    if (P == PP && N == NN) return sbf ? g.template go<PP, NN, StBF16>()      \
                                       : g.template go<PP, NN, StF32>();
    RSSM_M2S_CASE(64, 128)
    RSSM_M2S_CASE(128, 128)
    RSSM_M2S_CASE(64, 64)
    RSSM_M2S_CASE(128, 64)
#undef RSSM_M2S_CASE
    return RSSM_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" size_t rssm_mamba2_spec_workspace_size(const rssm_mamba2_dims* d, int32_t T) {
    if (m2::check_dims(d) || T < 1 || T > m2spec::kMaxT) return 0;
    return (size_t)d->batch * d->nheads * m2spec::tbl_floats(d->ring_len, T) * sizeof(float);
}

extern "C" int rssm_mamba2_spec_verify(const rssm_mamba2_dims* d, int32_t T, void* state,
                                       const void* x, const float* dt_raw, const float* dt_bias,
                                       int dt_softplus, const float* A, const void* B,
                                       const void* C, const float* D, const void* z,
                                       void* ring_x, float* ring_dt, void* ring_B,
                                       const int32_t* cache_indices, const int32_t* slot_cnt,
                                       const int32_t* slot_base, const uint8_t* slot_flush,
                                       void* workspace, size_t workspace_bytes, void* y,
                                       int32_t* dev_err, rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (T < 1 || T > m2spec::kMaxT || d->ring_len > 32) return RSSM_ERR_UNSUPPORTED;
    if (d->ring_len < 2 * T) return RSSM_ERR_CONFIG;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(x) || !ok_ptr(dt_raw) || !ok_opt_ptr(dt_bias) || !ok_ptr(A) ||
        !ok_ptr(B) || !ok_ptr(C) || !ok_ptr(D) || !ok_opt_ptr(z) || !ok_ptr(ring_x) ||
        !ok_ptr(ring_dt) || !ok_ptr(ring_B) || !ok_ptr(cache_indices) || !ok_ptr(slot_cnt) ||
        !ok_ptr(slot_base) || !ok_ptr(slot_flush) || !ok_ptr(workspace) || !ok_ptr(y))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_mamba2_spec_workspace_size(d, T)) return RSSM_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    switch (T) {
        case 1: return m2spec_launch<1>(d, state, x, dt_raw, dt_bias, dt_softplus, A, B, C, D, z,
                                        ring_x, ring_dt, ring_B, cache_indices, slot_cnt,
                                        slot_base, slot_flush, workspace, y, dev_err, st);
        case 2: return m2spec_launch<2>(d, state, x, dt_raw, dt_bias, dt_softplus, A, B, C, D, z,
                                        ring_x, ring_dt, ring_B, cache_indices, slot_cnt,
                                        slot_base, slot_flush, workspace, y, dev_err, st);
        case 3: return m2spec_launch<3>(d, state, x, dt_raw, dt_bias, dt_softplus, A, B, C, D, z,
                                        ring_x, ring_dt, ring_B, cache_indices, slot_cnt,
                                        slot_base, slot_flush, workspace, y, dev_err, st);
        default: return m2spec_launch<4>(d, state, x, dt_raw, dt_bias, dt_softplus, A, B, C, D, z,
                                         ring_x, ring_dt, ring_B, cache_indices, slot_cnt,
                                         slot_base, slot_flush, workspace, y, dev_err, st);
    }
}
