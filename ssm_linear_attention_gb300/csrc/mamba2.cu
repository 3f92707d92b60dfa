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

// ----------------------------------------------------------------------------
// output / flush kernel
// ----------------------------------------------------------------------------
//
// The producer copies a (row, head) checkpoint tile with 2-D TMA tensor copies and
// the 128-byte shared-memory swizzle: the tile is N * SS / 128 boxes of [P rows][128
// bytes], and row p's 16-byte chunk c lies at (c / 8) * P * 128 + p * 128 + 16 ((c % 8)
// ^ (p % 8)). The lanes of a quarter-warp then hit different banks both when they
// read different chunks of one row (the y dot products: 16 lanes per row) and when
// they read the same chunk of different rows (the flush: one row per lane).
// Tiles are claimed dynamically from a counter in the workspace: a flush tile costs
// several plain tiles, and with a static share the groups that drew more of them set
// the launch time.
//
// Flush rows fold the ring into the tile and write it back in place -- lane l of
// consumer warp wi owns tile row(s) p = 32 wi + l (+ 64), same swizzle -- and one
// thread stores the tile with TMA tensor stores. The fold is the product of
// A[p][i] = a_i x_i[p] and the ring's B entries:
//   * TC (64 x 128 tiles, bf16 ring, w + 1 <= 16): on the tensor cores. Each lane
//     writes Pm1 S0 of its row into its TMEM lane of the group's 128 accumulator
//     columns (M = 128: the group's 64 rows are the TMEM lanes its two warps may read,
//     64 (g % 2) .. +63; the other 64 rows are unused), the group stages A (float32,
//     three bf16 parts along K) and B^T in its scratch, one thread issues three
//     tcgen05.mma of K = 16 accumulating onto it, and each lane reads its row back.
//     Scratch of a pair of groups (4 warps x kTcWarpScratch):
//       [B^T of the even group][A of both groups: 16 row blocks x 768 B][B^T of odd]
//     so both groups' A descriptors start at the same address.
//   * otherwise (and for folds of fewer than kTcMinEntries entries, where the tensor
//     cores' fixed cost does not pay) on CUDA cores in the y mapping, stored from
//     registers with coalesced 16-byte stores.
template <int P, int N, class ST>
struct RowTile {
    static constexpr int SS = ST::bytes;
    static constexpr int TILE = P * N * SS;
    static constexpr int BOXC = 128 / SS;   // columns per 128-byte box row
    static constexpr int NBOX = N / BOXC;   // boxes per tile
    static constexpr int BOXB = P * 128;    // bytes per box
    static constexpr int CH = N * SS / 16;  // 16-byte chunks per row
    static constexpr int EPC = 16 / SS;     // elements per chunk
    static constexpr int RPL = P / 64;      // rows per lane (two warps of 32 lanes)
    static_assert(N % BOXC == 0 && P % 64 == 0, "tile shape");
    static __device__ __forceinline__ uint32_t off(int p, int c) {
        return (uint32_t)(c >> 3) * BOXB + (uint32_t)p * 128u + ((uint32_t)((c & 7) ^ (p & 7)) << 4);
    }
};

constexpr int kTcWarpScratch = 5120;
constexpr int kTcBT = 4096;            // B^T: 128 rows x 16 entries, bf16, core matrices
constexpr int kTcA = 16 * 768;         // A: 128 rows x 48 (3 parts x 16 entries), bf16
constexpr uint32_t kTcALbo = 128, kTcASbo = 768, kTcBLbo = 128, kTcBSbo = 256;
constexpr int kTcMaxEntries = 16;
constexpr int kTcMinEntries = 8;  // flushes of fewer entries take the CUDA-core fold

// The EPC elements of a 16-byte state chunk as float32.
template <class ST>
__device__ __forceinline__ void load_chunk(const uint8_t* p, float* f) {
    if constexpr (ST::bf16) {
        load8(p, true, f);
    } else {
        const float4 v = *reinterpret_cast<const float4*>(p);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
}

template <int P, int N, class ST, bool TC = false>
struct OutPolicy {
    using Rt = RowTile<P, N, ST>;
    static constexpr int kGroup = kGroupWarps;
    static constexpr int kTmemCols = TC ? 512 : 0;  // 128 accumulator columns per group
    static constexpr bool kUsesCtx = true;
    static constexpr bool kDynamic = true;  // tiles are claimed from a counter (flush tiles cost more)
    static_assert(!TC || (P == 64 && N == 128), "the tensor-core fold takes 64 x 128 tiles");
    struct Args {
        CUtensorMap tmap;  // the state pool as [slots * H * P rows][N], boxes of P x 128 bytes
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
        unsigned int* sched; // the work counter (workspace, after the tables)
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
        mbar_arrive_expect_tx(full, Rt::TILE + xbytes + N * sa + (a.z ? P * sa : 0) + TBL * 4 + bbytes);
        const int row0 = (m.s * a.H + h) * P;
#pragma unroll
        for (int bx = 0; bx < Rt::NBOX; ++bx)
            tma_load_2d(sb + bx * Rt::BOXB, &a.tmap, bx * Rt::BOXC, row0, full, pol);
        bulk_g2s(sb + a.off_x,
                 static_cast<const char*>(a.ring_x) + ((size_t)m.s * a.H + h) * a.L * P * sa, xbytes,
                 full);
        bulk_g2s(sb + a.off_C, static_cast<const char*>(a.C) + ((size_t)b * a.G + g) * N * sa, N * sa,
                 full);
        if (a.z)
            bulk_g2s(sb + a.off_z, static_cast<const char*>(a.z) + ((size_t)b * a.H + h) * P * sa,
                     P * sa, full);
        bulk_g2s(sb + a.off_tbl, a.ws + ((size_t)b * a.H + h) * TBL, TBL * 4, full);
        if (bbytes)
            bulk_g2s(sb + a.off_B,
                     static_cast<const char*>(a.ring_B) + ((size_t)m.s * a.G + g) * a.L * N * sa,
                     bbytes, full);
    }

    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb,
                                   uint8_t* scratch, int lane, int wi, PipeCtx& ctx) {
        if (!m.valid) return;
        const bool bf = a.act_bf16;
        const int L = a.L, w = m.w;
        const float* tbl = reinterpret_cast<const float*>(sb + a.off_tbl);
        const uint8_t* xr = sb + a.off_x;
        const uint8_t* Cs = sb + a.off_C;
        const float Pm1 = tbl[2 * L];
        const float Dh = __ldg(a.D + m.h);
        // y: 16 lanes (N = 128) share a row, each reading one 16-byte chunk of it (8
        // columns; two chunks for a float32 state) of RPI rows per load; the dot
        // products reduce across a row's lanes with reduce-scatters, after which every
        // lane holds whole results for NCH rows. The chunks a quarter-warp reads lie in
        // different banks under the swizzle.
        using Sh = TileShape<P, N, ST>;
        const int q = lane % Sh::NQ, hr = lane / Sh::NQ;
        const int row0 = wi * Sh::PW + hr;  // this lane's rows: row0 + RPI * t
        float part[Sh::ITER];
        if (ST::bf16 && bf) {
            const uint4 cpk = *reinterpret_cast<const uint4*>(Cs + q * 16);
#pragma unroll
            for (int t = 0; t < Sh::ITER; ++t) {
                const uint4 s8 = *reinterpret_cast<const uint4*>(sb + Rt::off(row0 + Sh::RPI * t, q));
                part[t] = dot8_bf16(s8, cpk, 0.f);
            }
        } else {
            float c[8];
            load8(Cs + q * 8 * (bf ? 2 : 4), bf, c);
#pragma unroll
            for (int t = 0; t < Sh::ITER; ++t) {
                const int p = row0 + Sh::RPI * t;
                float s8[8];
                if constexpr (ST::bf16) {
                    load8(sb + Rt::off(p, q), true, s8);
                } else {
                    load_chunk<ST>(sb + Rt::off(p, 2 * q), s8);
                    load_chunk<ST>(sb + Rt::off(p, 2 * q + 1), s8 + 4);
                }
                float acc = s8[0] * c[0];
#pragma unroll
                for (int j = 1; j < 8; ++j) acc = fmaf(s8[j], c[j], acc);
                part[t] = acc;
            }
        }
#pragma unroll
        for (int ch = 0; ch < Sh::NCH; ++ch) reduce_scatter<Sh::NQ, Sh::NQ>(part + ch * Sh::NQ);
#pragma unroll
        for (int ch = 0; ch < Sh::NCH; ++ch) {
            const int p = row0 + Sh::RPI * (ch * Sh::NQ + q);
            float yv = Pm1 * part[ch * Sh::NQ];
            float y2 = 0.f;
            int i = 0;
#pragma unroll 1
            for (; i + 1 <= w; i += 2) {
                yv = fmaf(tbl[i], load1(xr, i * P + p, bf), yv);
                y2 = fmaf(tbl[i + 1], load1(xr, (i + 1) * P + p, bf), y2);
            }
            if (i == w) yv = fmaf(tbl[w], load1(xr, w * P + p, bf), yv);
            yv += y2;
            yv = fmaf(Dh, load1(xr, w * P + p, bf), yv);
            if (a.z) yv *= silu_fast(load1(sb + a.off_z, p, bf));
            store1(a.y, ((size_t)m.b * a.H + m.h) * P + p, a.out_bf16, yv);
        }
        if (!m.f) return;
        if constexpr (TC) {
            // the tensor-core fold has a fixed cost; short rings fold faster on CUDA cores
            if (w + 1 >= kTcMinEntries) {
                fold_tc(a, m, const_cast<uint8_t*>(sb), scratch, lane, wi, ctx, tbl);
                store_tile(a, m, sb, lane, wi, ctx);
                return;
            }
        }
        fold_fma(a, m, sb, lane, wi, tbl);
    }

    // S = Pm1 S0 + sum_{i<=w} a_i x_i B_i^T on CUDA cores, in the y mapping (a lane owns 8
    // columns of rows row0 + RPI t), stored from registers: 16 lanes cover a row's
    // contiguous bytes, so the stores coalesce. Columns pairs accumulate with packed
    // two-wide FMAs.
    static __device__ void fold_fma(const Args& a, const Meta& m, const uint8_t* sb, int lane, int wi,
                                    const float* tbl) {
        using Sh = TileShape<P, N, ST>;
        const bool bf = a.act_bf16;
        const int sa = bf ? 2 : 4;
        const int L = a.L, w = m.w;
        const int q = lane % Sh::NQ, hr = lane / Sh::NQ;
        const int row0 = wi * Sh::PW + hr;
        const uint8_t* xr = sb + a.off_x;
        const uint8_t* br = sb + a.off_B;
        const float Pm1 = tbl[2 * L];
        const float* av = tbl + L;
        const size_t tile_e = ((size_t)m.s * a.H + m.h) * P * N;
        const ulonglong2 gen = load_generator<ST>(a.sr);
        constexpr int RC = Sh::ITER < 8 ? Sh::ITER : 8;
#pragma unroll 1
        for (int t0 = 0; t0 < Sh::ITER; t0 += RC) {
            float2 acc[RC][4];
#pragma unroll
            for (int r = 0; r < RC; ++r) {
                const int p = row0 + Sh::RPI * (t0 + r);
                float s8[8];
                if constexpr (ST::bf16) {
                    load8(sb + Rt::off(p, q), true, s8);
                } else {
                    load_chunk<ST>(sb + Rt::off(p, 2 * q), s8);
                    load_chunk<ST>(sb + Rt::off(p, 2 * q + 1), s8 + 4);
                }
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

    // One 16-byte chunk of a state row, rounded to the state dtype (stochastically for
    // StBF16SR, with the bits of the chunk's pool element index e), into the stage.
    static __device__ __forceinline__ void pack_chunk(uint8_t* dst, const float* f, size_t e,
                                                      ulonglong2 gen) {
        if constexpr (ST::bf16) {
            if constexpr (ST::sr) *reinterpret_cast<uint4*>(dst) = pack8_bf16_sr(f, e >> 3, gen.x, gen.y);
            else *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                                             pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
        } else {
            *reinterpret_cast<float4*>(dst) = make_float4(f[0], f[1], f[2], f[3]);
        }
    }

    static __device__ void fold_tc(const Args& a, const Meta& m, uint8_t* sb, uint8_t* scratch,
                                   int lane, int wi, PipeCtx& ctx, const float* tbl);

    // The folded tile (in the stage, written by both warps) to the pool with TMA tensor
    // stores; the issuing thread waits until they have read the stage and releases it
    // for both warps. The hand-over is a bounded mbarrier wait (not bar.sync), so a
    // group whose other warp left the loop on an abort cannot wait forever.
    // Warp 1 waits until the issuing thread has taken the hand-over ("taken" barrier),
    // so it can never arrive twice in one phase of the hand-over barrier.
    static __device__ void store_tile(const Args& a, const Meta& m, const uint8_t* sb, int lane, int wi,
                                      PipeCtx& ctx) {
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_plain(ctx.grp_bar);
        if (wi == 0 && lane == 0) {
            const bool ok = mbar_wait_bounded(ctx.grp_bar, ctx.grp_phase);
            if (ok) {
                const int row0 = (m.s * a.H + m.h) * P;
#pragma unroll
                for (int bx = 0; bx < Rt::NBOX; ++bx)
                    tma_store_2d(&a.tmap, bx * Rt::BOXC, row0, sb + bx * Rt::BOXB);
                bulk_commit();
            } else {
                *ctx.abort_flag = 1;
                set_dev_err(a.dev_err, RSSM_DEVERR_TIMEOUT);
            }
            mbar_arrive_plain(ctx.done_bar);
            if (ok) bulk_wait_read_all();
            mbar_arrive_count(ctx.empty_bar, kGroupWarps);  // the stage, for both warps
        }
        if (wi != 0 && !mbar_wait_bounded(ctx.done_bar, ctx.done_phase) && lane == 0) {
            *ctx.abort_flag = 1;
            set_dev_err(a.dev_err, RSSM_DEVERR_TIMEOUT);
        }
        ctx.grp_phase ^= 1;
        ctx.done_phase ^= 1;
        ctx.released = true;
    }
};

template <int P, int N, class ST, bool TC>
__device__ void OutPolicy<P, N, ST, TC>::fold_tc(const Args& a, const Meta& m, uint8_t* sb,
                                                 uint8_t* scratch, int lane, int wi, PipeCtx& ctx,
                                                 const float* tbl) {
    if constexpr (TC) {
        const int L = a.L, w = m.w;
        const int g = ctx.group;
        const int p = 32 * wi + lane;                  // this lane's tile row
        const int t = p;
        const uint32_t dcol = ctx.tmem + 128u * g;     // the group's accumulator columns
        const uint32_t lanes = (uint32_t)(64 * (g & 1) + 32 * wi) << 16;  // this warp's TMEM lanes
        const float Pm1 = tbl[2 * L];
        // 1. D = Pm1 S0 for this row, into TMEM (the group's previous MMA and this lane's
        //    previous TMEM reads are complete)
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32 / Rt::EPC; ++j)
                load_chunk<ST>(sb + Rt::off(p, c0 / Rt::EPC + j), v + Rt::EPC * j);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= Pm1;
            umma::st32(dcol + lanes + c0, v);
        }
        // 2. this row of A, a_i x_i[p] for i <= w (zero above), as three bf16 parts, into
        //    the pair's A rows; B^T blocks t < N / 4 (n-block nb, entry block kb) from the
        //    stage's ring rows (entries above w zero) into the group's B^T
        uint8_t* pair = scratch - wi * a.warp_scratch - (g & 1) * kGroupWarps * a.warp_scratch;
        uint8_t* Ab = pair + kTcBT;
        uint8_t* BT = (g & 1) ? pair + kTcBT + kTcA : pair;
        {
            const float* av = tbl + L;
            const uint16_t* xr = reinterpret_cast<const uint16_t*>(sb + a.off_x);
            uint16_t part[3][kTcMaxEntries];
#pragma unroll
            for (int i = 0; i < kTcMaxEntries; ++i) {
                float c = 0.f;
                if (i <= w) c = av[i] * bf16_to_f(xr[i * P + p]);
                umma::split3_bf16(c, part[0][i], part[1][i], part[2][i]);
            }
            const int arow = 64 * (g & 1) + p;
#pragma unroll
            for (int sp = 0; sp < 3; ++sp)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint16_t* q = &part[sp][8 * h];
                    *reinterpret_cast<uint4*>(Ab + umma::kmajor_offset(arow, 16 * sp + 8 * h, kTcALbo,
                                                                       kTcASbo)) =
                        make_uint4(q[0] | (uint32_t(q[1]) << 16), q[2] | (uint32_t(q[3]) << 16),
                                   q[4] | (uint32_t(q[5]) << 16), q[6] | (uint32_t(q[7]) << 16));
                }
        }
        if (t < N / 4) {
            const int nb = t % (N / 8), kb = t / (N / 8);
            const uint8_t* br = sb + a.off_B;
            uint4 in[8], out[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int e = 8 * kb + r;
                in[r] = e <= w ? *reinterpret_cast<const uint4*>(br + ((size_t)e * N + 8 * nb) * 2)
                               : make_uint4(0, 0, 0, 0);
            }
            umma::transpose8x8_b16(in, out);
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(BT + umma::kmajor_offset(8 * nb + c, 8 * kb, kTcBLbo, kTcBSbo)) =
                    out[c];
        }
        umma::wait_st();
        // 3. hand the operands to the issuing thread: writers fence their stores for the
        //    tensor core's (async) proxy and order their TMEM stores, then each warp
        //    arrives once (bounded wait, as in store_tile)
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_plain(ctx.grp_bar);
        if (t == 0) {
            if (mbar_wait_bounded(ctx.grp_bar, ctx.grp_phase)) {
                umma::fence_after_sync();
                constexpr uint32_t idesc = umma::idesc_bf16_f32(128, N);
                const uint64_t bdesc = umma::smem_desc_kmajor(BT, kTcBLbo, kTcBSbo);
#pragma unroll
                for (int sp = 0; sp < 3; ++sp)
                    umma::mma_bf16(dcol, umma::smem_desc_kmajor(Ab + sp * 2 * kTcALbo, kTcALbo, kTcASbo),
                                   bdesc, idesc, true);
                umma::commit_to(ctx.mma_bar);
            }
        }
        ctx.grp_phase ^= 1;
        const bool ok = mbar_wait_bounded(ctx.mma_bar, ctx.mma_phase);
        ctx.mma_phase ^= 1;
        umma::fence_after_sync();
        if (!ok) {
            if (lane == 0) {
                *ctx.abort_flag = 1;
                set_dev_err(a.dev_err, RSSM_DEVERR_TIMEOUT);
            }
            return;
        }
        // 4. the row back from TMEM, rounded to the state dtype, over S0 in the stage
        const size_t row_e = ((size_t)m.s * a.H + m.h) * P * N + (size_t)p * N;
        const ulonglong2 gen = load_generator<ST>(a.sr);
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 64) {
            float v[64];
            umma::ld64(dcol + lanes + c0, v);
            umma::wait_ld();
#pragma unroll
            for (int j = 0; j < 64 / Rt::EPC; ++j)
                pack_chunk(sb + Rt::off(p, c0 / Rt::EPC + j), v + Rt::EPC * j, row_e + c0 + Rt::EPC * j, gen);
        }
    }
}

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
            if (a.z) acc *= silu_fast(load1(sb + a.off_z, p, bf));
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
        // the tensor-core fold takes 64 x 128 tiles, bf16 ring entries and at most 16 of
        // them; rings too short to reach kTcMinEntries entries keep the leaner kernel
        if constexpr (P == 64 && N == 128) {
            if (!ST::sr && c.act_bf16 && c.L >= kTcMinEntries && c.L <= kTcMaxEntries)
                return run<OutPolicy<P, N, ST, true>, P, N>();
        }
        return run<OutPolicy<P, N, ST, false>, P, N>();
    }
    template <class Pol, int P, int N>
    int run() {
        typename Pol::Args a{};
        using Rt = typename Pol::Rt;
        if (!make_tmap_rows128(&a.tmap, c.state, Rt::SS, (uint64_t)c.num_slots * c.H * P, N, P))
            return RSSM_ERR_CUDA;
        a.state = c.state; a.C = c.C; a.D = c.D; a.z = c.z; a.ring_x = c.ring_x; a.ring_B = c.ring_B;
        a.ci = c.ci; a.row_wp = c.row_wp; a.row_flush = c.row_flush; a.ws = c.ws; a.y = c.y;
        a.dev_err = c.dev_err; a.sr = c.sr; a.batch = c.batch; a.H = c.H; a.G = c.G; a.L = c.L;
        a.num_slots = c.num_slots; a.act_bf16 = c.act_bf16; a.out_bf16 = c.out_bf16;
        a.sched = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(const_cast<float*>(c.ws)) +
                                                  sched_offset(c.batch, c.H, c.L));
        const int sa = c.act_bf16 ? 2 : 4;
        int off = Rt::TILE;
        a.off_x = off;   off += c.L * P * sa;
        a.off_C = off;   off += N * sa;
        a.off_z = off;   off += P * sa;
        a.off_tbl = off; off += tbl_floats(c.L) * 4;
        a.off_B = off;   off += c.L * N * sa;
        // 128-byte-swizzled boxes start on 1024-byte boundaries
        const int stage_bytes = (off + 1023) & ~1023;
        const int scratch = Pol::kTmemCols > 0 ? kTcWarpScratch : 0;
        return launch_pipe<Pol>(a, stage_bytes, scratch, Rt::TILE, (long)c.batch * c.H, stream, 1024);
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
    // a few rows: the whole step in one launch (round-to-nearest stores, cursor advanced here)
    if (sr_state == nullptr && advance && d->batch <= m2::kSmallStepMaxBatch &&
        d->ring_len <= m2::kSmallStepMaxRing) {
        if (!ok_ptr(x) || !ok_ptr(dt_raw) || !ok_opt_ptr(dt_bias) || !ok_ptr(A) || !ok_ptr(B) ||
            !ok_ptr(C) || !ok_ptr(cache_indices) || !ok_opt_ptr(force_flush) || !ok_ptr(slot_wp) ||
            !ok_ptr(row_wp) || !ok_ptr(ring_x) || !ok_ptr(ring_dt) || !ok_ptr(ring_B) ||
            !ok_ptr(workspace))
            return RSSM_ERR_INVALID_ARG;
        if (workspace_bytes < rssm_mamba2_workspace_size(d)) return RSSM_ERR_INVALID_ARG;
        rc = m2_step_small(d, force_flush, slot_wp, row_wp, row_flush, state, x, dt_raw, dt_bias,
                           dt_softplus, A, B, C, D, z, cache_indices, ring_x, ring_dt, ring_B,
                           workspace, y, dev_err, (cudaStream_t)stream);
        if (rc != RSSM_ERR_UNSUPPORTED) return rc;
    }
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
