// materialize.cu -- the full recurrent state of listed slots, folded from the
// checkpoint and the live ring entries into a separate fp32 buffer, without
// touching the pool, the rings or the cursors (test / debug entry points).
//
// Pages followed: [M2] "ReplaySSM: cache SSM inputs for faster Mamba2 standard
// decode", 实现拆解 item 1 (a flush writes back exactly the checkpoint advanced
// by the buffered steps); [GDN] "GDN ReplaySSM decode (Part A of RFC 28511)",
// 实现拆解 item 1 (the state every L steps is the checkpoint folded with the
// (d, k, g) ring); [SPEC] "[GDN] Support ReplaySSM Ring Spec-Verify", 实现拆解
// item 2 (the committed entries of a slot sit at cache_base .. cache_base+cnt-1 of
// the circular ring).
//
// Mamba2, slot s with c = slot_wp[s] live entries (0..c-1):
//   S = P S0 + sum_{i<c} P_i dt_i x_i B_i^T,  P_i = exp(A sum_{i<j<c} dt_j),
//   P = exp(A sum_{j<c} dt_j).
// GDN, slot s with c live entries at positions (base + i) % L:
//   S = G S0 + sum_{i<c} Gamma_i d_i k_i^T,  Gamma_i = prod_{i<j<c} g_j,
//   G = prod_{j<c} g_j.
// One CTA per (listed slot, head) or (listed slot, value head, 32-row block);
// plain loads and fp32 accumulation: these calls are not on the decode path.
#include "common.cuh"
#include "internal.h"
#include "gdn.cuh"
#include "mamba2.cuh"

namespace rssm {
namespace {

__global__ void m2_materialize_kernel(int H, int P, int N, int G, int L, int num_slots,
                                      int st_bf16, int act_bf16, const void* state,
                                      const float* A, const void* ring_x, const float* ring_dt,
                                      const void* ring_B, const int32_t* slots,
                                      const int32_t* slot_wp, float* out, int32_t* dev_err) {
    extern __shared__ float coef[];  // [L] P_i dt_i, then P
    const int j = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
    const int s = slots[j];
    if (s < 0) return;
    if (s >= num_slots) {
        if (threadIdx.x == 0 && h == 0) set_dev_err(dev_err, RSSM_DEVERR_SLOT);
        return;
    }
    const int c = slot_wp[s];
    if (c < 0 || c > L) {
        if (threadIdx.x == 0 && h == 0) set_dev_err(dev_err, RSSM_DEVERR_CURSOR);
        return;
    }
    if (threadIdx.x == 0) {
        const float* dt = ring_dt + ((size_t)s * H + h) * L;
        float suffix = 0.f;
        for (int i = c - 1; i >= 0; --i) {
            coef[i] = expf(A[h] * suffix) * dt[i];
            suffix += dt[i];
        }
        coef[L] = expf(A[h] * suffix);
    }
    __syncthreads();
    const int g = h / (H / G);
    const size_t tile = ((size_t)s * H + h) * P * N;
    for (int e = threadIdx.x; e < P * N; e += blockDim.x) {
        const int p = e / N, n = e - (e / N) * N;
        float acc = coef[L] * load1(state, (long)(tile + e), st_bf16);
        for (int i = 0; i < c; ++i) {
            const float xi = load1(ring_x, (long)((((size_t)s * H + h) * L + i) * P + p), act_bf16);
            const float bi = load1(ring_B, (long)((((size_t)s * G + g) * L + i) * N + n), act_bf16);
            acc = fmaf(coef[i] * xi, bi, acc);
        }
        out[((size_t)j * H + h) * P * N + e] = acc;
    }
}

__global__ void gdn_materialize_kernel(int HV, int HK, int V, int L, int num_slots, int act_bf16,
                                       const float* state, const void* ring_k, const float* ring_g,
                                       const float* ring_d, const int32_t* slots,
                                       const int32_t* slot_wp, const int32_t* slot_base,
                                       float* out, int32_t* dev_err) {
    extern __shared__ float gam[];  // [L] Gamma_i, then G
    const int NVB = V / gdn::VB;
    const int per = HV * NVB;
    const int j = blockIdx.x / per, rem = blockIdx.x - (blockIdx.x / per) * per;
    const int hv = rem / NVB, vb = rem - (rem / NVB) * NVB;
    const int s = slots[j];
    if (s < 0) return;
    const bool lead = threadIdx.x == 0 && rem == 0;
    if (s >= num_slots) {
        if (lead) set_dev_err(dev_err, RSSM_DEVERR_SLOT);
        return;
    }
    const int c = slot_wp[s], base = slot_base ? slot_base[s] : 0;
    if (c < 0 || c > L || base < 0 || base >= L) {
        if (lead) set_dev_err(dev_err, RSSM_DEVERR_CURSOR);
        return;
    }
    if (threadIdx.x == 0) {
        float p = 1.f;
        for (int i = c - 1; i >= 0; --i) {
            gam[i] = p;
            p *= ring_g[((size_t)s * HV + hv) * L + (base + i) % L];
        }
        gam[L] = p;
    }
    __syncthreads();
    const int kh = hv / (HV / HK);
    constexpr int KD = gdn::KD, VB = gdn::VB;
    const float* S0 = state + (((size_t)s * HV + hv) * V + (size_t)vb * VB) * KD;
    float* dst = out + (((size_t)j * HV + hv) * V + (size_t)vb * VB) * KD;
    for (int e = threadIdx.x; e < VB * KD; e += blockDim.x) {
        const int r = e / KD, kc = e - (e / KD) * KD;
        float acc = gam[L] * S0[e];
        for (int i = 0; i < c; ++i) {
            const int pos = (base + i) % L;
            const float di = ring_d[((((size_t)s * HV + hv) * NVB + vb) * L + pos) * VB + r];
            const float ki = load1(ring_k, (long)((((size_t)s * HK + kh) * L + pos) * KD + kc),
                                   act_bf16);
            acc = fmaf(gam[i] * di, ki, acc);
        }
        dst[e] = acc;
    }
}

}  // namespace
}  // namespace rssm

using namespace rssm;

extern "C" int rssm_mamba2_materialize_state(const rssm_mamba2_dims* d, const void* state,
                                             const float* A, const void* ring_x,
                                             const float* ring_dt, const void* ring_B,
                                             const int32_t* slots, const int32_t* slot_wp,
                                             float* out, int32_t* dev_err, rssm_stream_t stream) {
    int rc = m2::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(A) || !ok_ptr(ring_x) || !ok_ptr(ring_dt) || !ok_ptr(ring_B) ||
        !ok_ptr(slots) || !ok_ptr(slot_wp) || !ok_ptr(out))
        return RSSM_ERR_INVALID_ARG;
    const int smem = (d->ring_len + 1) * 4;
    if (smem > 48 * 1024) return RSSM_ERR_UNSUPPORTED;
    m2_materialize_kernel<<<d->batch * d->nheads, 256, smem, (cudaStream_t)stream>>>(
        d->nheads, d->headdim, d->dstate, d->ngroups, d->ring_len, d->num_slots,
        d->state_dtype == RSSM_BF16, d->act_dtype == RSSM_BF16, state, A, ring_x, ring_dt, ring_B,
        slots, slot_wp, out, dev_err);
    return launch_status();
}

extern "C" int rssm_gdn_materialize_state(const rssm_gdn_dims* d, const float* state,
                                          const void* ring_k, const float* ring_g,
                                          const float* ring_d, const int32_t* slots,
                                          const int32_t* slot_wp, const int32_t* slot_base,
                                          float* out, int32_t* dev_err, rssm_stream_t stream) {
    int rc = gdn::check_dims(d);
    if (rc) return rc;
    if (d->batch == 0) return RSSM_OK;
    if (!ok_ptr(state) || !ok_ptr(ring_k) || !ok_ptr(ring_g) || !ok_ptr(ring_d) || !ok_ptr(slots) ||
        !ok_ptr(slot_wp) || !ok_opt_ptr(slot_base) || !ok_ptr(out))
        return RSSM_ERR_INVALID_ARG;
    const int smem = (d->ring_len + 1) * 4;
    if (smem > 48 * 1024) return RSSM_ERR_UNSUPPORTED;
    const long blocks = (long)d->batch * d->num_v_heads * (d->head_v_dim / gdn::VB);
    gdn_materialize_kernel<<<(unsigned)blocks, 256, smem, (cudaStream_t)stream>>>(
        d->num_v_heads, d->num_k_heads, d->head_v_dim, d->ring_len, d->num_slots,
        d->act_dtype == RSSM_BF16, state, ring_k, ring_g, ring_d, slots, slot_wp, slot_base, out,
        dev_err);
    return launch_status();
}
