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
// Kernels (the per-row prologue kernels are in mamba2_prologue.cu):
//   output_kernel<P,N,ST> persistent, one work item = one (row, head) checkpoint
//                         tile. Per CTA several independent pipelines, each a
//                         producer warp feeding its own ring of shared-memory
//                         stages with 1-D TMA bulk copies (tile, ring x entries,
//                         C, z, table, and on flush rows the ring B entries)
//                         that complete on one mbarrier per stage, and a group of
//                         two consumer warps that reduce the tile against C with
//                         16-byte shared loads and warp reduce-scatters; flush
//                         rows fold the ring into the tile in registers and
//                         store it.
//   full_state_kernel<P,N,ST>  the conventional step (read tile, update, write
//                         tile, output) on the same pipeline.
#include <cstdio>

#include "common.cuh"
#include "internal.h"
#include "mamba2.cuh"
#include "pipeline.cuh"

namespace rssm {
namespace m2 {


// ----------------------------------------------------------------------------
// streaming kernels (warp-specialised pipeline, one consumer warp per tile)
// ----------------------------------------------------------------------------
//
// Tile (row b, head h): P x N state elements, consumed by a group of two warps
// that take half of the headdim rows each. A lane owns 8 consecutive dstate
// columns q = lane % (N/8) and every (32 / (N/8))-th row of its warp's half
// starting at lane / (N/8); one 16-byte shared load per lane covers 32 / (N/8)
// rows. Dot products over dstate reduce across the N/8 lanes of a row with
// reduce-scatters, after which every lane holds whole results for P/64 rows.
// With a bf16 state and bf16 C the products are mixed-precision fmas on the
// packed bf16 operands.

constexpr int kGroupWarps = 2;  // warps sharing one tile (half the headdim rows each)

template <int P, int N, class ST>
struct TileShape {
    static constexpr int SS = ST::bytes;
    static constexpr int TILE = P * N * SS;
    static constexpr int PW = P / kGroupWarps;  // rows per warp
    static constexpr int NQ = N / 8;            // lanes per row
    static constexpr int RPI = 32 / NQ;         // rows per load instruction
    static constexpr int ITER = PW / RPI;       // loads per lane
    static constexpr int NCH = ITER / NQ;       // rows per lane after the reduce-scatters
    static_assert(NCH >= 1 && ITER % NQ == 0, "tile shape");
};

// Store 8 state elements at element index e of the pool (e % 8 == 0): rounded to
// nearest, or (StBF16SR) stochastically with the bits of Philox4x32-10 at counter
// (e / 8, g.y), key g.x.
template <class ST>
__device__ __forceinline__ void store_state8(char* pool, size_t e, const float* f, ulonglong2 g) {
    void* p = pool + e * ST::bytes;
    if constexpr (ST::sr) store8_bf16_sr(p, f, e >> 3, g.x, g.y);
    else store8(p, ST::bf16, f);
}

// The generator {seed, offset} of a stochastically rounding launch, read once per
// tile before its stores (the state stores could alias it, so reading it inside the
// store loop would reload it every time).
template <class ST>
__device__ __forceinline__ ulonglong2 load_generator(const uint64_t* sr) {
    if constexpr (ST::sr) return make_ulonglong2(__ldg(sr), __ldg(sr + 1));
    else return make_ulonglong2(0, 0);
}

template <int P, int N, class ST>
struct OutPolicy {
    using Sh = TileShape<P, N, ST>;
    static constexpr int kGroup = kGroupWarps;
    struct Args {
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
        const uint64_t* sr;  // {seed, offset}: stochastic rounding of a bf16 state; null: nearest
        int batch, H, G, L, num_slots, act_bf16, out_bf16;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
        int off_x, off_C, off_z, off_tbl, off_B;
    };
    struct Meta {
        int valid, s, b, h, w, f;
    };

    static __device__ int n_items(const Args& a) { return a.batch * a.H; }

    static __device__ int4 prefetch(const Args& a, int item) {
        const int b = item / a.H;
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
        const int b = r.w, h = item - r.w * a.H;
        Meta m{0, r.x, b, h, r.y, r.z};
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
        const int g = h / (a.H / a.G);
        const int TBL = tbl_floats(a.L);
        const uint32_t xbytes = (m.w + 1) * P * sa;
        const uint32_t bbytes = m.f ? (m.w + 1) * N * sa : 0;
        mbar_arrive_expect_tx(full, Sh::TILE + xbytes + N * sa + (a.z ? P * sa : 0) + TBL * 4 + bbytes);
        bulk_g2s_hint(sb, static_cast<const char*>(a.state) + ((size_t)m.s * a.H + h) * Sh::TILE,
                      Sh::TILE, full, pol);
        bulk_g2s(sb + a.off_x,
                 static_cast<const char*>(a.ring_x) + ((size_t)m.s * a.H + h) * a.L * P * sa, xbytes,
                 full);
        bulk_g2s(sb + a.off_C, static_cast<const char*>(a.C) + ((size_t)b * a.G + g) * N * sa, N * sa,
                 full);
        if (a.z)
            bulk_g2s(sb + a.off_z, static_cast<const char*>(a.z) + ((size_t)b * a.H + h) * P * sa,
                     P * sa, full);
        bulk_g2s(sb + a.off_tbl, a.ws + ((size_t)b * a.H + h) * TBL, TBL * 4, full);
        if (m.f)
            bulk_g2s(sb + a.off_B,
                     static_cast<const char*>(a.ring_B) + ((size_t)m.s * a.G + g) * a.L * N * sa,
                     bbytes, full);
    }

    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb, uint8_t*,
                                   int lane, int wi) {
        if (!m.valid) return;
        const bool bf = a.act_bf16;
        const int sa = bf ? 2 : 4;
        const int L = a.L, w = m.w;
        const int q = lane % Sh::NQ, hr = lane / Sh::NQ;
        const int row0 = wi * Sh::PW + hr;  // this lane's rows: row0 + RPI * t
        const float* tbl = reinterpret_cast<const float*>(sb + a.off_tbl);
        const uint8_t* xr = sb + a.off_x;
        float part[Sh::ITER];
        if (ST::bf16 && bf) {
            const uint4 cpk = *reinterpret_cast<const uint4*>(sb + a.off_C + q * 16);
#pragma unroll
            for (int t = 0; t < Sh::ITER; ++t) {
                const int p = row0 + Sh::RPI * t;
                const uint4 s8 = *reinterpret_cast<const uint4*>(sb + ((size_t)p * N + q * 8) * Sh::SS);
                part[t] = dot8_bf16(s8, cpk, 0.f);
            }
        } else {
            float c[8];
            load8(sb + a.off_C + q * 8 * sa, bf, c);
#pragma unroll
            for (int t = 0; t < Sh::ITER; ++t) {
                const int p = row0 + Sh::RPI * t;
                float s8[8];
                load8(sb + ((size_t)p * N + q * 8) * Sh::SS, ST::bf16, s8);
                float acc = s8[0] * c[0];
#pragma unroll
                for (int j = 1; j < 8; ++j) acc = fmaf(s8[j], c[j], acc);
                part[t] = acc;
            }
        }
#pragma unroll
        for (int ch = 0; ch < Sh::NCH; ++ch) reduce_scatter<Sh::NQ, Sh::NQ>(part + ch * Sh::NQ);
        const float Pm1 = tbl[2 * L];
        const float Dh = __ldg(a.D + m.h);
#pragma unroll
        for (int ch = 0; ch < Sh::NCH; ++ch) {
            const int p = row0 + Sh::RPI * (ch * Sh::NQ + q);
            float acc = Pm1 * part[ch * Sh::NQ];
            float acc2 = 0.f;
            int i = 0;
#pragma unroll 1
            for (; i + 1 <= w; i += 2) {
                acc = fmaf(tbl[i], load1(xr, i * P + p, bf), acc);
                acc2 = fmaf(tbl[i + 1], load1(xr, (i + 1) * P + p, bf), acc2);
            }
            if (i == w) acc = fmaf(tbl[w], load1(xr, w * P + p, bf), acc);
            acc += acc2;
            acc = fmaf(Dh, load1(xr, w * P + p, bf), acc);
            if (a.z) acc *= silu_f(load1(sb + a.off_z, p, bf));
            store1(a.y, ((size_t)m.b * a.H + m.h) * P + p, a.out_bf16, acc);
        }
        if (m.f) {
            // S = Pm1 * S0 + sum_{i<=w} a_i x_i B_i^T, stored rounded to the state dtype
            const uint8_t* br = sb + a.off_B;
            const float* av = tbl + L;
            const size_t tile_e = ((size_t)m.s * a.H + m.h) * P * N;  // first element of the tile
            const ulonglong2 gen = load_generator<ST>(a.sr);
            constexpr int RC = Sh::ITER < 8 ? Sh::ITER : 8;
#pragma unroll 1
            for (int t0 = 0; t0 < Sh::ITER; t0 += RC) {
                // column pairs (2k, 2k+1) accumulate with packed two-wide FMAs
                float2 acc[RC][4];
#pragma unroll
                for (int r = 0; r < RC; ++r) {
                    const int p = row0 + Sh::RPI * (t0 + r);
                    float s8[8];
                    load8(sb + ((size_t)p * N + q * 8) * Sh::SS, ST::bf16, s8);
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
                        const int p = row0 + Sh::RPI * (t0 + r);
                        const float ax = ai * load1(xr, i * P + p, bf);
                        const float2 ax2 = make_float2(ax, ax);
#pragma unroll
                        for (int k = 0; k < 4; ++k) acc[r][k] = __ffma2_rn(ax2, b2[k], acc[r][k]);
                    }
                }
#pragma unroll
                for (int r = 0; r < RC; ++r) {
                    const int p = row0 + Sh::RPI * (t0 + r);
                    store_state8<ST>(static_cast<char*>(a.state), tile_e + (size_t)p * N + q * 8,
                                     reinterpret_cast<const float*>(acc[r]), gen);
                }
            }
        }
    }
};

template <int P, int N, class ST>
struct FullPolicy {
    using Sh = TileShape<P, N, ST>;
    static constexpr int kGroup = kGroupWarps;
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
        void* y;
        int32_t* dev_err;
        const uint64_t* sr;  // {seed, offset}: stochastic rounding of a bf16 state; null: nearest
        int batch, H, G, num_slots, act_bf16, out_bf16, softplus;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
        int off_x, off_B, off_C, off_z;
    };
    struct Meta {
        int valid, s, b, h;
        float dt, dA;
    };

    static __device__ int n_items(const Args& a) { return a.batch * a.H; }

    // dt = softplus(dt_raw + dt_bias) and dA = exp(A dt), computed by the producer lanes
    static __device__ int4 prefetch(const Args& a, int item) {
        const int b = item / a.H, h = item - (item / a.H) * a.H;
        const int s = a.ci[b];
        float dt = 0.f, dA = 0.f;
        if (s >= 0 && s < a.num_slots) {
            dt = a.dt_raw[(size_t)b * a.H + h] + (a.dt_bias ? a.dt_bias[h] : 0.f);
            if (a.softplus) dt = softplus_f(dt);
            dA = expf(a.A[h] * dt);
        }
        return make_int4(s, b, __float_as_int(dt), __float_as_int(dA));
    }

    static __device__ void issue(const Args& a, int item, int4 r, Meta* meta, uint8_t* sb,
                                 uint64_t* full, uint64_t pol) {
        const int b = r.y, h = item - r.y * a.H;
        Meta m{0, r.x, b, h, __int_as_float(r.z), __int_as_float(r.w)};
        if (r.x >= a.num_slots) set_dev_err(a.dev_err, RSSM_DEVERR_SLOT);
        else if (r.x >= 0) m.valid = 1;
        *meta = m;
        if (!m.valid) {
            mbar_arrive_plain(full);
            return;
        }
        const int sa = a.act_bf16 ? 2 : 4;
        const int g = h / (a.H / a.G);
        mbar_arrive_expect_tx(full, Sh::TILE + P * sa + 2 * N * sa + (a.z ? P * sa : 0));
        bulk_g2s_hint(sb, static_cast<const char*>(a.state) + ((size_t)m.s * a.H + h) * Sh::TILE,
                      Sh::TILE, full, pol);
        bulk_g2s(sb + a.off_x, static_cast<const char*>(a.x) + ((size_t)b * a.H + h) * P * sa, P * sa,
                 full);
        bulk_g2s(sb + a.off_B, static_cast<const char*>(a.B) + ((size_t)b * a.G + g) * N * sa, N * sa,
                 full);
        bulk_g2s(sb + a.off_C, static_cast<const char*>(a.C) + ((size_t)b * a.G + g) * N * sa, N * sa,
                 full);
        if (a.z)
            bulk_g2s(sb + a.off_z, static_cast<const char*>(a.z) + ((size_t)b * a.H + h) * P * sa,
                     P * sa, full);
    }

    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb, uint8_t*,
                                   int lane, int wi) {
        if (!m.valid) return;
        const bool bf = a.act_bf16;
        const int sa = bf ? 2 : 4;
        const int q = lane % Sh::NQ, hr = lane / Sh::NQ;
        const int row0 = wi * Sh::PW + hr;
        float c[8], bq[8];
        load8(sb + a.off_C + q * 8 * sa, bf, c);
        load8(sb + a.off_B + q * 8 * sa, bf, bq);
        const size_t tile_e = ((size_t)m.s * a.H + m.h) * P * N;  // first element of the tile
        const ulonglong2 gen = load_generator<ST>(a.sr);
        float part[Sh::ITER];
#pragma unroll
        for (int t = 0; t < Sh::ITER; ++t) {
            const int p = row0 + Sh::RPI * t;
            float s8[8];
            load8(sb + ((size_t)p * N + q * 8) * Sh::SS, ST::bf16, s8);
            const float dx = m.dt * load1(sb + a.off_x, p, bf);
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                s8[j] = fmaf(m.dA, s8[j], dx * bq[j]);
                acc = fmaf(s8[j], c[j], acc);
            }
            part[t] = acc;
            store_state8<ST>(static_cast<char*>(a.state), tile_e + (size_t)p * N + q * 8, s8, gen);
        }
#pragma unroll
        for (int ch = 0; ch < Sh::NCH; ++ch) reduce_scatter<Sh::NQ, Sh::NQ>(part + ch * Sh::NQ);
        const float Dh = __ldg(a.D + m.h);
#pragma unroll
        for (int ch = 0; ch < Sh::NCH; ++ch) {
            const int p = row0 + Sh::RPI * (ch * Sh::NQ + q);
            float acc = fmaf(Dh, load1(sb + a.off_x, p, bf), part[ch * Sh::NQ]);
            if (a.z) acc *= silu_f(load1(sb + a.off_z, p, bf));
            store1(a.y, ((size_t)m.b * a.H + m.h) * P + p, a.out_bf16, acc);
        }
    }
};

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


// sr: a bf16 state is stored with stochastic rounding (a float32 state ignores it).
template <class F>
int dispatch_pn(int P, int N, int state_dtype, bool sr, F&& f) {
#define RSSM_M2_CASE(PP, NN)                                                        \
    if (P == PP && N == NN) {                                                        \
        if (state_dtype == RSSM_BF16 && sr) return f.template go<PP, NN, StBF16SR>(); \
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

// Generic launch arguments, copied into each policy's Args by go<>().
struct OutCommon {
    void* state; const void* C; const float* D; const void* z; const void* ring_x; const void* ring_B;
    const int32_t* ci; const int32_t* row_wp; const uint8_t* row_flush; const float* ws; void* y;
    int32_t* dev_err; const uint64_t* sr; int batch, H, G, L, num_slots, act_bf16, out_bf16;
};

struct OutLaunch {
    OutCommon c;
    cudaStream_t stream;
    template <int P, int N, class ST>
    int go() {
        using Pol = OutPolicy<P, N, ST>;
        typename Pol::Args a{};
        a.state = c.state; a.C = c.C; a.D = c.D; a.z = c.z; a.ring_x = c.ring_x; a.ring_B = c.ring_B;
        a.ci = c.ci; a.row_wp = c.row_wp; a.row_flush = c.row_flush; a.ws = c.ws; a.y = c.y;
        a.dev_err = c.dev_err; a.sr = c.sr; a.batch = c.batch; a.H = c.H; a.G = c.G; a.L = c.L;
        a.num_slots = c.num_slots; a.act_bf16 = c.act_bf16; a.out_bf16 = c.out_bf16;
        const int sa = c.act_bf16 ? 2 : 4;
        int off = Pol::Sh::TILE;
        a.off_x = off;   off += c.L * P * sa;
        a.off_C = off;   off += N * sa;
        a.off_z = off;   off += P * sa;
        a.off_tbl = off; off += tbl_floats(c.L) * 4;
        a.off_B = off;   off += c.L * N * sa;
        const int stage_bytes = (off + 127) & ~127;
        return launch_pipe<Pol>(a, stage_bytes, 0, Pol::Sh::TILE, (long)c.batch * c.H, stream);
    }
};

struct FullCommon {
    void* state; const void* x; const float* dt_raw; const float* dt_bias; const float* A;
    const void* B; const void* C; const float* D; const void* z; const int32_t* ci; void* y;
    int32_t* dev_err; const uint64_t* sr; int batch, H, G, num_slots, act_bf16, out_bf16, softplus;
};

struct FullLaunch {
    FullCommon c;
    cudaStream_t stream;
    template <int P, int N, class ST>
    int go() {
        using Pol = FullPolicy<P, N, ST>;
        typename Pol::Args a{};
        a.state = c.state; a.x = c.x; a.dt_raw = c.dt_raw; a.dt_bias = c.dt_bias; a.A = c.A;
        a.B = c.B; a.C = c.C; a.D = c.D; a.z = c.z; a.ci = c.ci; a.y = c.y; a.dev_err = c.dev_err;
        a.sr = c.sr;
        a.batch = c.batch; a.H = c.H; a.G = c.G; a.num_slots = c.num_slots;
        a.act_bf16 = c.act_bf16; a.out_bf16 = c.out_bf16; a.softplus = c.softplus;
        const int sa = c.act_bf16 ? 2 : 4;
        int off = Pol::Sh::TILE;
        a.off_x = off; off += P * sa;
        a.off_B = off; off += N * sa;
        a.off_C = off; off += N * sa;
        a.off_z = off; off += P * sa;
        const int stage_bytes = (off + 127) & ~127;
        return launch_pipe<Pol>(a, stage_bytes, 0, Pol::Sh::TILE, (long)c.batch * c.H, stream);
    }
};

// The generator's offset moves on after each launch that drew from it, so the next
// launch (eager or replayed from a graph) draws fresh bits.
__global__ void sr_advance_kernel(uint64_t* sr) { sr[1] += 1; }

// out[4 g .. 4 g + 3] = Philox4x32-10 at counter (g, offset), key seed: the bits the
// stochastic rounding of 8-element group g draws (test / debug).
__global__ void philox_fill_kernel(uint64_t seed, uint64_t offset, uint32_t* out, size_t n) {
    const size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n) return;
    const uint4 r = philox4x32_10(
        make_uint4((uint32_t)g, (uint32_t)(g >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)),
        make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
    reinterpret_cast<uint4*>(out)[g] = r;
}

}  // namespace m2
}  // namespace rssm

using namespace rssm;

namespace {

int m2_output_impl(const rssm_mamba2_dims* d, void* state, const void* C, const float* D,
                   const void* z, const void* ring_x, const void* ring_B,
                   const int32_t* cache_indices, const int32_t* row_wp, const uint8_t* row_flush,
                   const void* workspace, size_t workspace_bytes, void* y, int32_t* dev_err,
                   uint64_t* sr, rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(C) || !ok_ptr(D) || !ok_opt_ptr(z) || !ok_ptr(ring_x) ||
        !ok_ptr(ring_B) || !ok_ptr(cache_indices) || !ok_ptr(row_wp) || !ok_ptr(row_flush) ||
        !ok_ptr(workspace) || !ok_ptr(y) || !ok_opt_ptr(sr))
        return RSSM_ERR_INVALID_ARG;
    if (workspace_bytes < rssm_mamba2_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
    m2::OutLaunch l{};
    l.stream = (cudaStream_t)stream;
    m2::OutCommon& a = l.c;
    a.state = state; a.C = C; a.D = D; a.z = z; a.ring_x = ring_x; a.ring_B = ring_B;
    a.ci = cache_indices; a.row_wp = row_wp; a.row_flush = row_flush;
    a.ws = static_cast<const float*>(workspace); a.y = y; a.dev_err = dev_err; a.sr = sr;
    a.batch = d->batch; a.H = d->nheads; a.G = d->ngroups; a.L = d->ring_len;
    a.num_slots = d->num_slots; a.act_bf16 = d->act_dtype == RSSM_BF16;
    a.out_bf16 = d->out_dtype == RSSM_BF16;
    rc = m2::dispatch_pn(d->headdim, d->dstate, d->state_dtype, sr != nullptr, l);
    if (rc || sr == nullptr) return rc;
    m2::sr_advance_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(sr);
    return launch_status();
}

int m2_full_impl(const rssm_mamba2_dims* d, void* state, const void* x, const float* dt_raw,
                 const float* dt_bias, int dt_softplus, const float* A, const void* B,
                 const void* C, const float* D, const void* z, const int32_t* cache_indices,
                 void* y, int32_t* dev_err, uint64_t* sr, rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(x) || !ok_ptr(dt_raw) || !ok_opt_ptr(dt_bias) || !ok_ptr(A) ||
        !ok_ptr(B) || !ok_ptr(C) || !ok_ptr(D) || !ok_opt_ptr(z) || !ok_ptr(cache_indices) ||
        !ok_ptr(y) || !ok_opt_ptr(sr))
        return RSSM_ERR_INVALID_ARG;
    m2::FullLaunch l{};
    l.stream = (cudaStream_t)stream;
    m2::FullCommon& a = l.c;
    a.state = state; a.x = x; a.dt_raw = dt_raw; a.dt_bias = dt_bias; a.A = A; a.B = B; a.C = C;
    a.D = D; a.z = z; a.ci = cache_indices; a.y = y; a.dev_err = dev_err; a.sr = sr;
    a.batch = d->batch; a.H = d->nheads; a.G = d->ngroups; a.num_slots = d->num_slots;
    a.act_bf16 = d->act_dtype == RSSM_BF16; a.out_bf16 = d->out_dtype == RSSM_BF16;
    a.softplus = dt_softplus != 0;
    rc = m2::dispatch_pn(d->headdim, d->dstate, d->state_dtype, sr != nullptr, l);
    if (rc || sr == nullptr) return rc;
    m2::sr_advance_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(sr);
    return launch_status();
}

}  // namespace

extern "C" int rssm_mamba2_output(const rssm_mamba2_dims* d, void* state, const void* C,
                                  const float* D, const void* z, const void* ring_x,
                                  const void* ring_B, const int32_t* cache_indices,
                                  const int32_t* row_wp, const uint8_t* row_flush,
                                  const void* workspace, size_t workspace_bytes, void* y,
                                  int32_t* dev_err, rssm_stream_t stream) {
    return m2_output_impl(d, state, C, D, z, ring_x, ring_B, cache_indices, row_wp, row_flush,
                          workspace, workspace_bytes, y, dev_err, nullptr, stream);
}

extern "C" int rssm_mamba2_output_sr(const rssm_mamba2_dims* d, void* state, const void* C,
                                     const float* D, const void* z, const void* ring_x,
                                     const void* ring_B, const int32_t* cache_indices,
                                     const int32_t* row_wp, const uint8_t* row_flush,
                                     const void* workspace, size_t workspace_bytes, void* y,
                                     uint64_t* sr_state, int32_t* dev_err, rssm_stream_t stream) {
    if (!ok_ptr(sr_state)) return RSSM_ERR_INVALID_ARG;
    return m2_output_impl(d, state, C, D, z, ring_x, ring_B, cache_indices, row_wp, row_flush,
                          workspace, workspace_bytes, y, dev_err, sr_state, stream);
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

extern "C" int rssm_mamba2_step(const rssm_mamba2_dims* d, int advance, const uint8_t* force_flush,
                                int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush, void* state,
                                const void* x, const float* dt_raw, const float* dt_bias,
                                int dt_softplus, const float* A, const void* B, const void* C,
                                const float* D, const void* z, const int32_t* cache_indices,
                                void* ring_x, float* ring_dt, void* ring_B, void* workspace,
                                size_t workspace_bytes, void* y, int32_t* dev_err,
                                rssm_stream_t stream) {
    return rssm_mamba2_step_sr(d, advance, force_flush, slot_wp, row_wp, row_flush, state, x,
                               dt_raw, dt_bias, dt_softplus, A, B, C, D, z, cache_indices, ring_x,
                               ring_dt, ring_B, workspace, workspace_bytes, y, nullptr, dev_err,
                               stream);
}

extern "C" int rssm_mamba2_step_sr(const rssm_mamba2_dims* d, int advance,
                                   const uint8_t* force_flush, int32_t* slot_wp, int32_t* row_wp,
                                   uint8_t* row_flush, void* state, const void* x,
                                   const float* dt_raw, const float* dt_bias, int dt_softplus,
                                   const float* A, const void* B, const void* C, const float* D,
                                   const void* z, const int32_t* cache_indices, void* ring_x,
                                   float* ring_dt, void* ring_B, void* workspace,
                                   size_t workspace_bytes, void* y, uint64_t* sr_state,
                                   int32_t* dev_err, rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(D) || !ok_opt_ptr(z) || !ok_ptr(y) || !ok_ptr(row_flush) ||
        !ok_opt_ptr(sr_state))
        return RSSM_ERR_INVALID_ARG;
    rc = rssm_mamba2_prepare(d, advance, force_flush, slot_wp, row_wp, row_flush, x, dt_raw, dt_bias,
                             dt_softplus, B, A, C, cache_indices, ring_x, ring_dt, ring_B,
                             workspace, workspace_bytes, dev_err, stream);
    if (rc) return rc;
    return m2_output_impl(d, state, C, D, z, ring_x, ring_B, cache_indices, row_wp, row_flush,
                          workspace, workspace_bytes, y, dev_err, sr_state, stream);
}

extern "C" int rssm_mamba2_full_state_update(const rssm_mamba2_dims* d, void* state, const void* x,
                                             const float* dt_raw, const float* dt_bias,
                                             int dt_softplus, const float* A, const void* B,
                                             const void* C, const float* D, const void* z,
                                             const int32_t* cache_indices, void* y,
                                             int32_t* dev_err, rssm_stream_t stream) {
    return m2_full_impl(d, state, x, dt_raw, dt_bias, dt_softplus, A, B, C, D, z, cache_indices, y,
                        dev_err, nullptr, stream);
}

extern "C" int rssm_mamba2_full_state_update_sr(const rssm_mamba2_dims* d, void* state,
                                                const void* x, const float* dt_raw,
                                                const float* dt_bias, int dt_softplus,
                                                const float* A, const void* B, const void* C,
                                                const float* D, const void* z,
                                                const int32_t* cache_indices, void* y,
                                                uint64_t* sr_state, int32_t* dev_err,
                                                rssm_stream_t stream) {
    if (!ok_ptr(sr_state)) return RSSM_ERR_INVALID_ARG;
    return m2_full_impl(d, state, x, dt_raw, dt_bias, dt_softplus, A, B, C, D, z, cache_indices, y,
                        dev_err, sr_state, stream);
}

extern "C" int rssm_philox4x32_fill(uint64_t seed, uint64_t offset, uint32_t* out, size_t n_groups,
                                    rssm_stream_t stream) {
    if (n_groups == 0) return RSSM_OK;
    if (!ok_ptr(out)) return RSSM_ERR_INVALID_ARG;
    const unsigned blocks = (unsigned)((n_groups + 255) / 256);
    m2::philox_fill_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(seed, offset, out, n_groups);
    return launch_status();
}
