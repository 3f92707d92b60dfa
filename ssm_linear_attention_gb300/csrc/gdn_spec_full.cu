// gdn_spec_full.cu -- the conventional speculative verify for the gated delta net,
// built as the in-house comparison for the ReplaySSM verify (sm_103a).
//
// Pages followed: [SPEC] "[GDN] Support ReplaySSM Ring Spec-Verify" (SGLang PR
// 28695 report): 功能与动机 (the recurrent verify keeps a full-state snapshot per
// draft token, the intermediate_ssm buffers, which dominate spec-decode memory;
// the accepted draft's snapshot becomes the slot's state). The recurrence is the
// gated delta rule of [GDN] "GDN ReplaySSM decode (Part A of RFC 28511)":
//   S <- g S + beta (v - g S k) k^T,  o = S q.
//
// verify: one work item = (row, value head, 32-row block) of the slot's state,
// streamed once through the warp-specialised pipeline; the T drafts are applied
// in order to the tile in shared memory, draft j's output is written and the
// tile after draft j is stored as snapshot j. The pool is not modified.
// commit: for rows with a > 0 accepted drafts, snapshot a-1 is copied into the
// slot (a plain 16-byte copy kernel).
#include "common.cuh"
#include "gdn.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace rssm {
namespace specfull {

using gdn::KD;
using gdn::TILE;
using gdn::VB;
constexpr int kGroupWarps = 2;
constexpr int RW = VB / kGroupWarps;  // value rows per warp

template <int T>
struct Policy {
    static constexpr int kGroup = kGroupWarps;
    struct Args {
        const float* state;
        const void* q;
        const void* k;
        const void* v;
        const float* beta;
        const float* g;
        const int32_t* ci;
        float* snap;  // [batch][T][HV][V][K]
        void* o;      // [batch][T][HV][V]
        int32_t* dev_err;
        int batch, HV, HK, V, num_slots, act_bf16, out_bf16;
        int stages, stage_bytes, stage_off, scratch_off, warp_scratch;
        int off_kq, off_v;
    };
    struct Meta {
        int valid, s, b, hv, vb;
    };

    static __device__ int n_items(const Args& a) { return a.batch * a.HV * (a.V / VB); }

    static __device__ int4 prefetch(const Args& a, int item) {
        const int b = item / (a.HV * (a.V / VB));
        return make_int4(a.ci[b], b, 0, 0);
    }

    static __device__ void issue(const Args& a, int item, int4 r, Meta* meta, uint8_t* sb,
                                 uint64_t* full, uint64_t pol) {
        const int NVB = a.V / VB;
        const int b = r.y;
        const int rem = item - b * a.HV * NVB;
        const int hv = rem / NVB, vb = rem - (rem / NVB) * NVB;
        Meta m{0, r.x, b, hv, vb};
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
        mbar_arrive_expect_tx(full, TILE + 2 * T * kb + T * VB * sa);
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
    }

    // Each warp owns 16 value rows of the tile; lane l holds key columns 4l..4l+3.
    // Per draft: one 32-way reduce-scatter gives S k_j and S q_j for the 16 rows,
    // then d = beta (v - g S k), o = g (S q) + d (k . q), S = g S + d k^T (in shared
    // memory, rows private to the warp), and the rows go to snapshot j.
    static __device__ void consume(const Args& a, int, const Meta& m, const uint8_t* sb, uint8_t*,
                                   int lane, int wi) {
        if (!m.valid) return;
        const bool bf = a.act_bf16;
        const int sa = bf ? 2 : 4;
        float* tile = reinterpret_cast<float*>(const_cast<uint8_t*>(sb)) + wi * RW * KD;
        const uint8_t* kq = sb + a.off_kq;
        float bj = 0.f, gj = 0.f;
        if (lane < T) {
            bj = a.beta[((size_t)m.b * T + lane) * a.HV + m.hv];
            gj = a.g[((size_t)m.b * T + lane) * a.HV + m.hv];
        }
#pragma unroll 1
        for (int j = 0; j < T; ++j) {
            const float be = __shfl_sync(kFull, bj, j), ge = __shfl_sync(kFull, gj, j);
            float k4[4], q4[4];
            load4(kq + (size_t)(2 * j) * KD * sa, lane * 4, bf, k4);
            load4(kq + (size_t)(2 * j + 1) * KD * sa, lane * 4, bf, q4);
            float kqd = k4[0] * q4[0] + k4[1] * q4[1] + k4[2] * q4[2] + k4[3] * q4[3];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) kqd += __shfl_xor_sync(kFull, kqd, o);
            float part[32];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float4 s4 = *reinterpret_cast<const float4*>(tile + r * KD + lane * 4);
                part[r] = s4.x * k4[0] + s4.y * k4[1] + s4.z * k4[2] + s4.w * k4[3];
                part[16 + r] = s4.x * q4[0] + s4.y * q4[1] + s4.z * q4[2] + s4.w * q4[3];
            }
            reduce_scatter<32, 32>(part);  // lane l holds entry l: S k (l < 16), S q (l >= 16)
            const float sq = __shfl_down_sync(kFull, part[0], 16);
            float dn = 0.f;
            const int rr = wi * RW + (lane & 15);
            if (lane < 16) {
                dn = be * (load1(sb + a.off_v + j * VB * sa, rr, bf) - ge * part[0]);
                const float oo = ge * sq + dn * kqd;
                store1(a.o, (((size_t)m.b * T + j) * a.HV + m.hv) * a.V + (size_t)m.vb * VB + rr,
                       a.out_bf16, oo);
            }
            float* snap = a.snap + (((((size_t)m.b * T + j) * a.HV + m.hv) * a.V +
                                     (size_t)m.vb * VB + wi * RW) * KD);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float dr = __shfl_sync(kFull, dn, r);
                float4 s4 = *reinterpret_cast<const float4*>(tile + r * KD + lane * 4);
                s4.x = fmaf(ge, s4.x, dr * k4[0]);
                s4.y = fmaf(ge, s4.y, dr * k4[1]);
                s4.z = fmaf(ge, s4.z, dr * k4[2]);
                s4.w = fmaf(ge, s4.w, dr * k4[3]);
                *reinterpret_cast<float4*>(tile + r * KD + lane * 4) = s4;
                *reinterpret_cast<float4*>(snap + r * KD + lane * 4) = s4;
            }
            __syncwarp();
        }
    }
};

// Copy snapshot a-1 into the slot for rows with a > 0 accepted drafts. Grid: rows x
// chunks of 4096 floats.
__global__ void commit_kernel(int T, int HV, int V, int num_slots, const int32_t* ci,
                              const int32_t* acc, const float* snap, float* state,
                              int32_t* dev_err) {
    const size_t per = (size_t)HV * V * KD;  // floats per slot
    const int chunks = (int)(per / 4096);
    const int b = blockIdx.x / chunks, c = blockIdx.x - (blockIdx.x / chunks) * chunks;
    const int s = ci[b];
    if (s < 0) return;
    if (s >= num_slots) {
        if (threadIdx.x == 0 && c == 0) set_dev_err(dev_err, RSSM_DEVERR_SLOT);
        return;
    }
    const int n = acc[b];
    if (n < 0 || n > T) {
        if (threadIdx.x == 0 && c == 0) set_dev_err(dev_err, RSSM_DEVERR_CURSOR);
        return;
    }
    if (n == 0) return;
    const float4* src = reinterpret_cast<const float4*>(snap + ((size_t)b * T + (n - 1)) * per) +
                        (size_t)c * 1024;
    float4* dst = reinterpret_cast<float4*>(state + (size_t)s * per) + (size_t)c * 1024;
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) dst[i] = src[i];
}

template <int T>
int launch_verify(const rssm_gdn_dims* d, const float* state, const void* q, const void* k,
                  const void* v, const float* beta, const float* g, const int32_t* ci, float* snap,
                  void* o, int32_t* dev_err, cudaStream_t st) {
    const int sa = d->act_dtype == RSSM_BF16 ? 2 : 4;
    typename Policy<T>::Args a{};
    a.state = state; a.q = q; a.k = k; a.v = v; a.beta = beta; a.g = g; a.ci = ci; a.snap = snap;
    a.o = o; a.dev_err = dev_err;
    a.batch = d->batch; a.HV = d->num_v_heads; a.HK = d->num_k_heads; a.V = d->head_v_dim;
    a.num_slots = d->num_slots; a.act_bf16 = d->act_dtype == RSSM_BF16;
    a.out_bf16 = d->out_dtype == RSSM_BF16;
    int off = TILE;
    a.off_kq = off; off += 2 * T * KD * sa;
    a.off_v = off;  off += T * VB * sa;
    const int stage_bytes = (off + 127) & ~127;
    return launch_pipe<Policy<T>>(a, stage_bytes, 0, TILE,
                                  (long)d->batch * d->num_v_heads * (d->head_v_dim / VB), st);
}

int check(const rssm_gdn_dims* d, int T) {
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (T < 1) return RSSM_ERR_CONFIG;
    if (T > 8) return RSSM_ERR_UNSUPPORTED;
    return RSSM_OK;
}

}  // namespace specfull
}  // namespace rssm

using namespace rssm;

extern "C" size_t rssm_gdn_spec_full_state_snapshot_bytes(const rssm_gdn_dims* d, int32_t T) {
    if (specfull::check(d, T)) return 0;
    return (size_t)d->batch * T * d->num_v_heads * d->head_v_dim * d->head_k_dim * sizeof(float);
}

extern "C" int rssm_gdn_spec_full_state_verify(const rssm_gdn_dims* d, int32_t T,
                                               const float* state, const void* q, const void* k,
                                               const void* v, const float* beta, const float* g,
                                               const int32_t* cache_indices, float* snapshots,
                                               size_t snapshot_bytes, void* o, int32_t* dev_err,
                                               rssm_stream_t stream) {
    int rc = specfull::check(d, T);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(beta) || !ok_ptr(g) ||
        !ok_ptr(cache_indices) || !ok_ptr(snapshots) || !ok_ptr(o))
        return RSSM_ERR_INVALID_ARG;
    if (snapshot_bytes < rssm_gdn_spec_full_state_snapshot_bytes(d, T)) return RSSM_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    switch (T) {
        case 1: return specfull::launch_verify<1>(d, state, q, k, v, beta, g, cache_indices, snapshots, o, dev_err, st);
        case 2: return specfull::launch_verify<2>(d, state, q, k, v, beta, g, cache_indices, snapshots, o, dev_err, st);
        case 3: return specfull::launch_verify<3>(d, state, q, k, v, beta, g, cache_indices, snapshots, o, dev_err, st);
        case 4: return specfull::launch_verify<4>(d, state, q, k, v, beta, g, cache_indices, snapshots, o, dev_err, st);
        case 5: return specfull::launch_verify<5>(d, state, q, k, v, beta, g, cache_indices, snapshots, o, dev_err, st);
        case 6: return specfull::launch_verify<6>(d, state, q, k, v, beta, g, cache_indices, snapshots, o, dev_err, st);
        case 7: return specfull::launch_verify<7>(d, state, q, k, v, beta, g, cache_indices, snapshots, o, dev_err, st);
        default: return specfull::launch_verify<8>(d, state, q, k, v, beta, g, cache_indices, snapshots, o, dev_err, st);
    }
}

extern "C" int rssm_gdn_spec_full_state_commit(const rssm_gdn_dims* d, int32_t T, float* state,
                                               const float* snapshots,
                                               const int32_t* cache_indices,
                                               const int32_t* num_accepted, int32_t* dev_err,
                                               rssm_stream_t stream) {
    int rc = specfull::check(d, T);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(snapshots) || !ok_ptr(cache_indices) || !ok_ptr(num_accepted))
        return RSSM_ERR_INVALID_ARG;
    const long chunks = (long)d->num_v_heads * d->head_v_dim * specfull::KD / 4096;
    specfull::commit_kernel<<<(unsigned)(d->batch * chunks), 256, 0, (cudaStream_t)stream>>>(
        T, d->num_v_heads, d->head_v_dim, d->num_slots, cache_indices, num_accepted, snapshots,
        state, dev_err);
    return launch_status();
}
