/*
 * oracle.c -- float64 CPU oracle for ReplaySSM decode (Mamba2 and gated delta net).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark load this library. The CUDA product path never links, includes or
 * calls anything here, and nothing here is shared with it.
 *
 * Sources followed (the four web pages on ReplaySSM; the pages print no equations,
 * so the recurrences below are the textbook forms of the operations they name):
 *
 *   [M2]   "ReplaySSM: cache SSM inputs for faster Mamba2 standard decode"
 *          (vLLM PR 48018 report), sections 功能与动机 (motivation), 实现拆解
 *          (implementation breakdown) and 关键源码片段 (key source snippet: the
 *          baseline selective_state_update(ssm_state, x, dt, A, B, C, D, dt_bias,
 *          dt_softplus, state_batch_indices, out) call and the ReplaySSM call with
 *          x_cache, dt_cache, B_cache, write_pos, is_flush).
 *   [GDN]  "GDN ReplaySSM decode (Part A of RFC 28511)" (SGLang PR 28451 report),
 *          sections 功能与动机 and 实现拆解 item 1 (output reconstructed from the
 *          checkpoint S0 plus the (d, k, g) ring; full state flushed every L steps).
 *   [SPEC] "[GDN] Support ReplaySSM Ring Spec-Verify" (SGLang PR 28695 report),
 *          实现拆解 items 2-4 (per-draft outputs from checkpoint + circular ring; the
 *          exact fold replays the recurrent update from the raw inputs).
 *
 * Every function computes in double precision with plain loops in the order the
 * definition states. No blocking, no fusion, no reordering beyond the definition.
 * Parallelism is over independent batch rows only (POSIX threads).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------- */
/* Storage rounding (the "storage-faithful" mode)                            */
/* ------------------------------------------------------------------------- */

/* Round a double to the nearest bfloat16 value, ties to even.
 * bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and float32's exponent
 * range. frexp gives v = m * 2^e with 0.5 <= |m| < 1; scaling m by 2^8 puts the
 * kept bits left of the binary point, and nearbyint (default rounding mode: to
 * nearest, ties to even) rounds the rest away. Values below the float32 normal
 * range are rounded on the subnormal grid 2^-133. Overflow is not handled (the
 * workloads stay far below 3.4e38). */
double orc_round_bf16(double v) {
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    double m = frexp(v, &e);            /* v = m * 2^e */
    if (e - 8 < -133) {                 /* bf16 subnormal spacing is 2^-133 */
        return ldexp(nearbyint(ldexp(v, 133)), -133);
    }
    return ldexp(nearbyint(ldexp(m, 8)), e - 8);
}

/* Round a double to float32, ties to even (the C conversion under the default
 * rounding mode). */
double orc_round_f32(double v) { return (double)(float)v; }

/* softplus(x) = log(1 + e^x), written so that e^x never overflows:
 * for x > 0, log(1 + e^x) = x + log(1 + e^-x). */
double orc_softplus(double x) {
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Round every element of the listed slots of a slot-indexed pool to the storage
 * dtype (1 = float32, 2 = bfloat16). slot_elems = elements per slot. A negative
 * slot index is skipped. */
void orc_round_slots(double* pool, long slot_elems, const int* slots, int n, int dtype) {
    for (int i = 0; i < n; ++i) {
        if (slots[i] < 0) continue;
        double* p = pool + (long)slots[i] * slot_elems;
        for (long j = 0; j < slot_elems; ++j)
            p[j] = dtype == 2 ? orc_round_bf16(p[j]) : orc_round_f32(p[j]);
    }
}

/* ------------------------------------------------------------------------- */
/* Stochastic rounding of the bf16 state                                      */
/* ------------------------------------------------------------------------- */

/* [M2] 评论区精华: quantised models (the NVFP4 Nemotron baseline) rely on
 * stochastic rounding (SR) of the bf16 state, and the report adds SR as an option.
 * The pages give neither the generator nor the rounding rule; the library's
 * interface fixes both, and this is that definition written out.
 *
 * Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 * 1, 2, 3", SC 2011, section 3): a 4 x 32-bit counter and a 2 x 32-bit key; each of
 * the 10 rounds multiplies counter words 0 and 2 by the two Philox constants,
 * splits each 64-bit product into high and low halves, and outputs
 *   (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0));
 * between rounds the key is bumped by the two Weyl constants (golden ratio and
 * sqrt(3) - 1, times 2^32). */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint64_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = M0 * (uint64_t)c0;
        uint64_t p1 = M1 * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Stochastic rounding of v to bfloat16 with 16 random bits r (0 <= r < 2^16).
 * v is first taken to float32 (the precision the decode kernels accumulate the
 * state in, so that both sides decide in the same precision). With lo = the bf16
 * value next to v toward zero, u = the bf16 spacing there and
 * f = (|v| - |lo|) / u in [0, 1) (a multiple of 2^-16 for a float32 v), the result
 * is the neighbour away from zero when r + 2^16 f >= 2^16, else lo. Over all 2^16
 * values of r it rounds away from zero exactly 2^16 f times, so its mean is v.
 * 0, NaN and +-Inf are returned unchanged. */
double orc_round_bf16_sr(double v, unsigned r) {
    v = (double)(float)v;
    if (v == 0.0 || !isfinite(v)) return v;
    double a = fabs(v);
    int e;
    frexp(a, &e);                               /* a = m * 2^e, 0.5 <= m < 1 */
    int ue = e - 8 < -133 ? -133 : e - 8;       /* bf16 spacing 2^ue (subnormals 2^-133) */
    double u = ldexp(1.0, ue);
    double lo = floor(a / u) * u;
    double f = (a - lo) / u;
    double q = (double)(r & 0xFFFFu) + ldexp(f, 16) >= 65536.0 ? lo + u : lo;
    return v < 0 ? -q : q;
}

/* The 16 bits element e of a pool draws at generator (seed, offset): Philox
 * counter {e / 8 low word, e / 8 high word, offset low, offset high}, key {seed
 * low, seed high}; element j = e % 8 takes the low (j even) or high (j odd) half of
 * output word j / 2. */
unsigned orc_sr_bits(uint64_t seed, uint64_t offset, uint64_t e) {
    uint64_t g = e / 8;
    uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), (uint32_t)offset,
                       (uint32_t)(offset >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    unsigned j = (unsigned)(e % 8);
    uint32_t word = w[j / 2];
    return (j % 2 == 0 ? word : word >> 16) & 0xFFFFu;
}

/* Stochastically round every element of the listed slots of a slot-indexed pool
 * to bf16: element j of slot s has pool index e = s * slot_elems + j and draws
 * orc_sr_bits(seed, offset, e). A negative slot index is skipped. */
void orc_round_slots_sr(double* pool, long slot_elems, const int* slots, int n, uint64_t seed,
                        uint64_t offset) {
    for (int i = 0; i < n; ++i) {
        if (slots[i] < 0) continue;
        for (long j = 0; j < slot_elems; ++j) {
            uint64_t e = (uint64_t)slots[i] * (uint64_t)slot_elems + (uint64_t)j;
            double* p = pool + e;
            *p = orc_round_bf16_sr(*p, orc_sr_bits(seed, offset, e));
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Row-parallel driver                                                       */
/* ------------------------------------------------------------------------- */

typedef void (*row_fn)(const void* ctx, int b);
typedef struct { row_fn fn; const void* ctx; int batch; int tid; int nthreads; } worker_arg;

static void* worker(void* p) {
    worker_arg* a = (worker_arg*)p;
    for (int b = a->tid; b < a->batch; b += a->nthreads) a->fn(a->ctx, b);
    return NULL;
}

int orc_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void for_rows(row_fn fn, const void* ctx, int batch, int nthreads) {
    if (nthreads <= 0) nthreads = orc_default_threads();
    if (nthreads > batch) nthreads = batch > 0 ? batch : 1;
    if (nthreads == 1) {
        for (int b = 0; b < batch; ++b) fn(ctx, b);
        return;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
    worker_arg* args = (worker_arg*)malloc(sizeof(worker_arg) * nthreads);
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn; args[t].ctx = ctx; args[t].batch = batch;
        args[t].tid = t; args[t].nthreads = nthreads;
        pthread_create(&th[t], NULL, worker, &args[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th); free(args);
}

/* ------------------------------------------------------------------------- */
/* Mamba2: full-state recurrence (the conventional decode step)              */
/* ------------------------------------------------------------------------- */

typedef struct { int batch, nheads, headdim, dstate, ngroups, num_slots; } orc_m2_dims;

typedef struct {
    const orc_m2_dims* d;
    double* state;
    const double *x, *dt_raw, *dt_bias, *A, *B, *C, *D, *z;
    int dt_softplus;
    const int* ci;
    double* y;
} m2_step_ctx;

/* One decode step of the Mamba2 selective state update, for one row b.
 * [M2] key source snippet, baseline branch: selective_state_update(ssm_state, x,
 * dt, A, B, C, D, dt_bias, dt_softplus, state_batch_indices, out) reads and
 * writes the full state h[nheads, headdim, dstate] of slot ci[b]. Textbook form:
 *   dt   = softplus(dt_raw + dt_bias[h])           (when dt_softplus)
 *   dA   = exp(A[h] * dt)
 *   h[p][n] <- dA * h[p][n] + dt * x[p] * B[g][n]   (g = group of head h)
 *   y[p]  = sum_n h[p][n] * C[g][n] + D[h] * x[p]
 *   y[p] *= silu(z[p])                            (when z is given)
 * Heads are split into ngroups contiguous blocks of nheads/ngroups heads; all
 * heads of a block share B and C. */
static void m2_step_row(const void* vctx, int b) {
    const m2_step_ctx* c = (const m2_step_ctx*)vctx;
    const orc_m2_dims* d = c->d;
    const int H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups;
    const int s = c->ci[b];
    if (s < 0 || s >= d->num_slots) return;
    const int heads_per_group = H / G;
    for (int h = 0; h < H; ++h) {
        const int g = h / heads_per_group;
        double dt = c->dt_raw[(long)b * H + h] + (c->dt_bias ? c->dt_bias[h] : 0.0);
        if (c->dt_softplus) dt = orc_softplus(dt);
        const double dA = exp(c->A[h] * dt);
        double* hs = c->state + (((long)s * H + h) * P) * N;
        const double* Bg = c->B + ((long)b * G + g) * N;
        const double* Cg = c->C + ((long)b * G + g) * N;
        for (int p = 0; p < P; ++p) {
            const double xp = c->x[((long)b * H + h) * P + p];
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                double v = dA * hs[(long)p * N + n] + dt * xp * Bg[n];
                hs[(long)p * N + n] = v;
                acc += v * Cg[n];
            }
            double yp = acc + c->D[h] * xp;
            if (c->z) yp *= silu(c->z[((long)b * H + h) * P + p]);
            c->y[((long)b * H + h) * P + p] = yp;
        }
    }
}

int orc_mamba2_step(const orc_m2_dims* d, double* state, const double* x,
                    const double* dt_raw, const double* dt_bias, int dt_softplus,
                    const double* A, const double* B, const double* C, const double* D,
                    const double* z, const int* ci, double* y, int nthreads) {
    if (d->ngroups <= 0 || d->nheads % d->ngroups) return 3;
    m2_step_ctx c = {d, state, x, dt_raw, dt_bias, A, B, C, D, z, dt_softplus, ci, y};
    for_rows(m2_step_row, &c, d->batch, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Mamba2: ReplaySSM closed form (checkpoint + ring)                          */
/* ------------------------------------------------------------------------- */

typedef struct {
    const orc_m2_dims* d;
    int L;
    const double* S0;
    const int *ci, *wp;
    const double *ex, *edt_raw, *dt_bias, *A, *eB, *C, *D, *z;
    int dt_softplus;
    double *y, *S_fold;
} m2_replay_ctx;

/* Output of the current step computed from the frozen checkpoint S0 of the slot
 * and the ring entries 0..w (entry w is the current step), without forming the
 * state. [M2] 功能与动机: most steps read their output from checkpoint + buffer;
 * the full state is written back only every L steps. Unrolling the recurrence
 * above from S0 over entries i = 0..w gives, with dA_i = exp(A[h] * dt_i):
 *   y[p] = (prod_{j=0..w} dA_j) * sum_n S0[p][n] C[n]
 *        + sum_{i=0..w} (prod_{j=i+1..w} dA_j) * dt_i * x_i[p] * (B_i . C)
 *        + D[h] * x_w[p]
 *   gated by silu(z[p]);
 * and the folded state (the flush)
 *   S[p][n] = (prod_{j=0..w} dA_j) S0[p][n]
 *           + sum_{i=0..w} (prod_{j=i+1..w} dA_j) dt_i x_i[p] B_i[n].
 * Entry arrays are per row: ex[b][i][H][P], edt_raw[b][i][H], eB[b][i][G][N].
 * C is the current step's C[b][G][N]; z is the current z[b][H][P] or NULL.
 * S_fold (nullable) receives [batch][H][P][N]. */
static void m2_replay_row(const void* vctx, int b) {
    const m2_replay_ctx* c = (const m2_replay_ctx*)vctx;
    const orc_m2_dims* d = c->d;
    const int H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups, L = c->L;
    const int s = c->ci[b];
    if (s < 0 || s >= d->num_slots) return;
    const int w = c->wp[b];
    const int hpg = H / G;
    double* dt = (double*)malloc(sizeof(double) * (w + 1));
    double* dA = (double*)malloc(sizeof(double) * (w + 1));
    double* suffix = (double*)malloc(sizeof(double) * (w + 2)); /* suffix[i] = prod_{j=i..w} dA_j */
    double* bc = (double*)malloc(sizeof(double) * (w + 1));
    for (int h = 0; h < H; ++h) {
        const int g = h / hpg;
        for (int i = 0; i <= w; ++i) {
            double t = c->edt_raw[((long)b * L + i) * H + h] + (c->dt_bias ? c->dt_bias[h] : 0.0);
            dt[i] = c->dt_softplus ? orc_softplus(t) : t;
            dA[i] = exp(c->A[h] * dt[i]);
        }
        suffix[w + 1] = 1.0;
        for (int i = w; i >= 0; --i) suffix[i] = suffix[i + 1] * dA[i];
        const double* Cg = c->C + ((long)b * G + g) * N;
        for (int i = 0; i <= w; ++i) {
            const double* Bi = c->eB + (((long)b * L + i) * G + g) * N;
            double acc = 0.0;
            for (int n = 0; n < N; ++n) acc += Bi[n] * Cg[n];
            bc[i] = acc;
        }
        const double* S0h = c->S0 + (((long)s * H + h) * P) * N;
        for (int p = 0; p < P; ++p) {
            double s0c = 0.0;
            for (int n = 0; n < N; ++n) s0c += S0h[(long)p * N + n] * Cg[n];
            double yp = suffix[0] * s0c;
            for (int i = 0; i <= w; ++i) {
                const double xi = c->ex[(((long)b * L + i) * H + h) * P + p];
                yp += suffix[i + 1] * dt[i] * xi * bc[i];
            }
            const double xw = c->ex[(((long)b * L + w) * H + h) * P + p];
            yp += c->D[h] * xw;
            if (c->z) yp *= silu(c->z[((long)b * H + h) * P + p]);
            c->y[((long)b * H + h) * P + p] = yp;
            if (c->S_fold) {
                double* Sf = c->S_fold + (((long)b * H + h) * P) * N;
                for (int n = 0; n < N; ++n) {
                    double v = suffix[0] * S0h[(long)p * N + n];
                    for (int i = 0; i <= w; ++i) {
                        const double xi = c->ex[(((long)b * L + i) * H + h) * P + p];
                        const double Bin = c->eB[(((long)b * L + i) * G + g) * N + n];
                        v += suffix[i + 1] * dt[i] * xi * Bin;
                    }
                    Sf[(long)p * N + n] = v;
                }
            }
        }
    }
    free(dt); free(dA); free(suffix); free(bc);
}

int orc_mamba2_replay(const orc_m2_dims* d, int L, const double* S0, const int* ci,
                      const int* wp, const double* ex, const double* edt_raw,
                      const double* dt_bias, int dt_softplus, const double* A,
                      const double* eB, const double* C, const double* D, const double* z,
                      double* y, double* S_fold, int nthreads) {
    if (d->ngroups <= 0 || d->nheads % d->ngroups) return 3;
    for (int b = 0; b < d->batch; ++b)
        if (ci[b] >= 0 && (wp[b] < 0 || wp[b] >= L)) return 1;
    m2_replay_ctx c = {d, L, S0, ci, wp, ex, edt_raw, dt_bias, A, eB, C, D, z, dt_softplus, y, S_fold};
    for_rows(m2_replay_row, &c, d->batch, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Mamba2: one speculative verify round                                       */
/* ------------------------------------------------------------------------- */

typedef struct {
    const orc_m2_dims* d;
    int T;
    double* state;
    const double *x, *dt_raw, *dt_bias, *A, *B, *C, *D, *z;
    int dt_softplus;
    const int *ci, *acc;
    double* y;
} m2_spec_ctx;

/* The speculative round of the full ReplaySSM design ("ReplaySSM: cache SSM inputs
 * for faster Mamba2 standard decode", 关联脉络: PR 47576 covers Mamba2 and GDN,
 * standard and speculative decode), read the way the GDN spec verify page states
 * it: draft j's output is the recurrence's output after the committed history and
 * drafts 0..j (rejected drafts included); the commit keeps the state after the
 * first acc[b] drafts (acc in 0..T). Inputs per row and draft: x [b][T][H][P],
 * dt_raw [b][T][H], B, C [b][T][G][N], z [b][T][H][P] or NULL; y receives
 * [b][T][H][P]. Each head runs on a private copy of its state tile. */
static void m2_spec_row(const void* vctx, int b) {
    const m2_spec_ctx* c = (const m2_spec_ctx*)vctx;
    const orc_m2_dims* d = c->d;
    const int H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups, T = c->T;
    const int s = c->ci[b];
    if (s < 0 || s >= d->num_slots) return;
    const int acc = c->acc[b];
    const int hpg = H / G;
    double* S = (double*)malloc(sizeof(double) * (long)P * N);
    for (int h = 0; h < H; ++h) {
        const int g = h / hpg;
        double* Sslot = c->state + (((long)s * H + h) * P) * N;
        memcpy(S, Sslot, sizeof(double) * (long)P * N);
        for (int j = 0; j < T; ++j) {
            const long bj = (long)b * T + j;
            double dt = c->dt_raw[bj * H + h] + (c->dt_bias ? c->dt_bias[h] : 0.0);
            if (c->dt_softplus) dt = orc_softplus(dt);
            const double dA = exp(c->A[h] * dt);
            const double* Bg = c->B + (bj * G + g) * N;
            const double* Cg = c->C + (bj * G + g) * N;
            for (int p = 0; p < P; ++p) {
                const double xp = c->x[(bj * H + h) * P + p];
                double a = 0.0;
                for (int n = 0; n < N; ++n) {
                    const double v = dA * S[(long)p * N + n] + dt * xp * Bg[n];
                    S[(long)p * N + n] = v;
                    a += v * Cg[n];
                }
                double yp = a + c->D[h] * xp;
                if (c->z) yp *= silu(c->z[(bj * H + h) * P + p]);
                c->y[(bj * H + h) * P + p] = yp;
            }
            if (j + 1 == acc) memcpy(Sslot, S, sizeof(double) * (long)P * N);
        }
    }
    free(S);
}

int orc_mamba2_spec_round(const orc_m2_dims* d, int T, double* state, const double* x,
                          const double* dt_raw, const double* dt_bias, int dt_softplus,
                          const double* A, const double* B, const double* C, const double* D,
                          const double* z, const int* ci, const int* acc, double* y,
                          int nthreads) {
    if (d->ngroups <= 0 || d->nheads % d->ngroups) return 3;
    for (int b = 0; b < d->batch; ++b)
        if (ci[b] >= 0 && (acc[b] < 0 || acc[b] > T)) return 1;
    m2_spec_ctx c = {d, T, state, x, dt_raw, dt_bias, A, B, C, D, z, dt_softplus, ci, acc, y};
    for_rows(m2_spec_row, &c, d->batch, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Gated delta net: full-state recurrence                                    */
/* ------------------------------------------------------------------------- */

typedef struct { int batch, num_v_heads, num_k_heads, head_k_dim, head_v_dim, num_slots; } orc_gdn_dims;

/* The gated delta rule for one value head, in place on S[V][K]:
 *   u    = S k                 (u[v] = sum_k S[v][k] k[k])
 *   d    = beta * (v - g * u)
 *   S   <- g * S + d k^T
 *   o    = S q
 * This is S <- g S + beta (v - g S k) k^T, o = S q: the per-step read and write
 * of the full state [HV, V, K] that [GDN] 功能与动机 describes for the
 * conventional decode kernel. d is written to dout when dout is not NULL. */
static void gdn_head_step(double* S, int K, int V, const double* q, const double* k,
                          const double* v, double beta, double g, double* o, double* dout) {
    for (int iv = 0; iv < V; ++iv) {
        double u = 0.0;
        for (int ik = 0; ik < K; ++ik) u += S[(long)iv * K + ik] * k[ik];
        const double dv = beta * (v[iv] - g * u);
        if (dout) dout[iv] = dv;
        double acc = 0.0;
        for (int ik = 0; ik < K; ++ik) {
            const double nv = g * S[(long)iv * K + ik] + dv * k[ik];
            S[(long)iv * K + ik] = nv;
            acc += nv * q[ik];
        }
        if (o) o[iv] = acc;
    }
}

typedef struct {
    const orc_gdn_dims* d;
    double* state;
    const double *q, *k, *v, *beta, *g;
    const int* ci;
    double* o;
} gdn_step_ctx;

/* Value head hv reads key head hv / (HV / HK): contiguous blocks of value heads
 * share one key head (grouped-query layout, 2:1 in the pages' workload). */
static void gdn_step_row(const void* vctx, int b) {
    const gdn_step_ctx* c = (const gdn_step_ctx*)vctx;
    const orc_gdn_dims* d = c->d;
    const int HV = d->num_v_heads, HK = d->num_k_heads, K = d->head_k_dim, V = d->head_v_dim;
    const int s = c->ci[b];
    if (s < 0 || s >= d->num_slots) return;
    const int vpk = HV / HK;
    for (int hv = 0; hv < HV; ++hv) {
        const int kh = hv / vpk;
        double* S = c->state + (((long)s * HV + hv) * V) * K;
        gdn_head_step(S, K, V, c->q + ((long)b * HK + kh) * K, c->k + ((long)b * HK + kh) * K,
                      c->v + ((long)b * HV + hv) * V, c->beta[(long)b * HV + hv],
                      c->g[(long)b * HV + hv], c->o + ((long)b * HV + hv) * V, NULL);
    }
}

int orc_gdn_step(const orc_gdn_dims* d, double* state, const double* q, const double* k,
                 const double* v, const double* beta, const double* g, const int* ci,
                 double* o, int nthreads) {
    if (d->num_k_heads <= 0 || d->num_v_heads % d->num_k_heads) return 3;
    gdn_step_ctx c = {d, state, q, k, v, beta, g, ci, o};
    for_rows(gdn_step_row, &c, d->batch, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Gated delta net: ReplaySSM closed form (checkpoint + (d, k, g) ring)      */
/* ------------------------------------------------------------------------- */

typedef struct {
    const orc_gdn_dims* d;
    int L;
    const double* S0;
    const int *ci, *wp;
    const double *ek, *ev, *ebeta, *eg, *q;
    double *o, *S_fold, *d_out;
} gdn_replay_ctx;

/* [GDN] 实现拆解 item 1: a non-flush step reconstructs its output from the
 * checkpoint S0 and the ring of (d_i, k_i, g_i); the full state is only formed
 * at a flush. With entries i = 0..w (entry w is the current step) and
 * S^(i) = g_i S^(i-1) + d_i k_i^T, S^(-1) = S0, unrolling gives
 *   S^(i-1) k_i = (prod_{j<i} g_j) S0 k_i + sum_{m<i} (prod_{j=m+1..i-1} g_j) d_m (k_m . k_i)
 *   d_i         = beta_i (v_i - g_i S^(i-1) k_i)
 *   o_w = S^(w) q = (prod_{j<=w} g_j) S0 q + sum_{m<=w} (prod_{j=m+1..w} g_j) d_m (k_m . q)
 *   S^(w) = (prod_{j<=w} g_j) S0 + sum_{m<=w} (prod_{j=m+1..w} g_j) d_m k_m^T   (the flush)
 * The d_i are produced in order, each from the reconstruction (not from a
 * materialised state). Entry arrays per row: ek[b][i][HK][K], ev[b][i][HV][V],
 * ebeta[b][i][HV], eg[b][i][HV]; q is the current q[b][HK][K]. Outputs: o[b][HV][V];
 * S_fold (nullable) [b][HV][V][K]; d_out (nullable) [b][i][HV][V]. */
static void gdn_replay_row(const void* vctx, int b) {
    const gdn_replay_ctx* c = (const gdn_replay_ctx*)vctx;
    const orc_gdn_dims* d = c->d;
    const int HV = d->num_v_heads, HK = d->num_k_heads, K = d->head_k_dim, V = d->head_v_dim;
    const int L = c->L;
    const int s = c->ci[b];
    if (s < 0 || s >= d->num_slots) return;
    const int w = c->wp[b];
    const int vpk = HV / HK;
    double* dd = (double*)malloc(sizeof(double) * (long)(w + 1) * V);
    double* gk = (double*)malloc(sizeof(double) * (w + 1));
    double* tmp = (double*)malloc(sizeof(double) * V);
    for (int hv = 0; hv < HV; ++hv) {
        const int kh = hv / vpk;
        const double* S0 = c->S0 + (((long)s * HV + hv) * V) * K;
        for (int i = 0; i <= w; ++i) gk[i] = c->eg[((long)b * L + i) * HV + hv];
        /* d_i for i = 0..w, in order */
        for (int i = 0; i <= w; ++i) {
            const double* ki = c->ek + (((long)b * L + i) * HK + kh) * K;
            double G = 1.0;
            for (int j = 0; j < i; ++j) G *= gk[j];
            for (int iv = 0; iv < V; ++iv) {
                double s0k = 0.0;
                for (int ik = 0; ik < K; ++ik) s0k += S0[(long)iv * K + ik] * ki[ik];
                tmp[iv] = G * s0k;
            }
            for (int m = 0; m < i; ++m) {
                const double* km = c->ek + (((long)b * L + m) * HK + kh) * K;
                double kk = 0.0;
                for (int ik = 0; ik < K; ++ik) kk += km[ik] * ki[ik];
                double gam = 1.0;
                for (int j = m + 1; j < i; ++j) gam *= gk[j];
                for (int iv = 0; iv < V; ++iv) tmp[iv] += gam * dd[(long)m * V + iv] * kk;
            }
            const double be = c->ebeta[((long)b * L + i) * HV + hv];
            const double* vi = c->ev + (((long)b * L + i) * HV + hv) * V;
            for (int iv = 0; iv < V; ++iv) dd[(long)i * V + iv] = be * (vi[iv] - gk[i] * tmp[iv]);
        }
        /* o_w from S0 and the d, k, g entries */
        const double* q = c->q + ((long)b * HK + kh) * K;
        double Gall = 1.0;
        for (int j = 0; j <= w; ++j) Gall *= gk[j];
        for (int iv = 0; iv < V; ++iv) {
            double s0q = 0.0;
            for (int ik = 0; ik < K; ++ik) s0q += S0[(long)iv * K + ik] * q[ik];
            tmp[iv] = Gall * s0q;
        }
        for (int m = 0; m <= w; ++m) {
            const double* km = c->ek + (((long)b * L + m) * HK + kh) * K;
            double kq = 0.0;
            for (int ik = 0; ik < K; ++ik) kq += km[ik] * q[ik];
            double gam = 1.0;
            for (int j = m + 1; j <= w; ++j) gam *= gk[j];
            for (int iv = 0; iv < V; ++iv) tmp[iv] += gam * dd[(long)m * V + iv] * kq;
        }
        for (int iv = 0; iv < V; ++iv) c->o[((long)b * HV + hv) * V + iv] = tmp[iv];
        if (c->d_out)
            for (int i = 0; i <= w; ++i)
                for (int iv = 0; iv < V; ++iv)
                    c->d_out[(((long)b * L + i) * HV + hv) * V + iv] = dd[(long)i * V + iv];
        if (c->S_fold) {
            double* Sf = c->S_fold + (((long)b * HV + hv) * V) * K;
            for (int iv = 0; iv < V; ++iv)
                for (int ik = 0; ik < K; ++ik) {
                    double val = Gall * S0[(long)iv * K + ik];
                    for (int m = 0; m <= w; ++m) {
                        double gam = 1.0;
                        for (int j = m + 1; j <= w; ++j) gam *= gk[j];
                        const double km = c->ek[(((long)b * L + m) * HK + kh) * K + ik];
                        val += gam * dd[(long)m * V + iv] * km;
                    }
                    Sf[(long)iv * K + ik] = val;
                }
        }
    }
    free(dd); free(gk); free(tmp);
}

int orc_gdn_replay(const orc_gdn_dims* d, int L, const double* S0, const int* ci, const int* wp,
                   const double* ek, const double* ev, const double* ebeta, const double* eg,
                   const double* q, double* o, double* S_fold, double* d_out, int nthreads) {
    if (d->num_k_heads <= 0 || d->num_v_heads % d->num_k_heads) return 3;
    for (int b = 0; b < d->batch; ++b)
        if (ci[b] >= 0 && (wp[b] < 0 || wp[b] >= L)) return 1;
    gdn_replay_ctx c = {d, L, S0, ci, wp, ek, ev, ebeta, eg, q, o, S_fold, d_out};
    for_rows(gdn_replay_row, &c, d->batch, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* KDA: the gated delta rule with a per-key-channel gate                      */
/* ------------------------------------------------------------------------- */

/* [GDN] 实现拆解 item 1 builds one decode kernel for both the scalar-gate GDN and
 * the KDA per-K gate (IS_KDA); its 评论区精华 gives the KDA gate ring as
 * g_cache [slots, HV, L, K]. The pages state no equation; the reading here is the
 * gated delta rule with the scalar gate g replaced by a diagonal gate Diag(a),
 * a in (0, 1]^K, acting on the key channels of S[V][K]:
 *   u    = S Diag(a) k        (u[v] = sum_k S[v][k] a[k] k[k])
 *   d    = beta * (v - u)
 *   S   <- S Diag(a) + d k^T
 *   o    = S q
 * With a = g * 1 this is gdn_head_step. */
static void kda_head_step(double* S, int K, int V, const double* q, const double* k,
                          const double* v, double beta, const double* a, double* o,
                          double* dout) {
    for (int iv = 0; iv < V; ++iv) {
        double u = 0.0;
        for (int ik = 0; ik < K; ++ik) u += S[(long)iv * K + ik] * a[ik] * k[ik];
        const double dv = beta * (v[iv] - u);
        if (dout) dout[iv] = dv;
        double acc = 0.0;
        for (int ik = 0; ik < K; ++ik) {
            const double nv = S[(long)iv * K + ik] * a[ik] + dv * k[ik];
            S[(long)iv * K + ik] = nv;
            acc += nv * q[ik];
        }
        if (o) o[iv] = acc;
    }
}

typedef struct {
    const orc_gdn_dims* d;
    double* state;
    const double *q, *k, *v, *beta, *a;
    const int* ci;
    double* o;
} kda_step_ctx;

static void kda_step_row(const void* vctx, int b) {
    const kda_step_ctx* c = (const kda_step_ctx*)vctx;
    const orc_gdn_dims* d = c->d;
    const int HV = d->num_v_heads, HK = d->num_k_heads, K = d->head_k_dim, V = d->head_v_dim;
    const int s = c->ci[b];
    if (s < 0 || s >= d->num_slots) return;
    const int vpk = HV / HK;
    for (int hv = 0; hv < HV; ++hv) {
        const int kh = hv / vpk;
        double* S = c->state + (((long)s * HV + hv) * V) * K;
        kda_head_step(S, K, V, c->q + ((long)b * HK + kh) * K, c->k + ((long)b * HK + kh) * K,
                      c->v + ((long)b * HV + hv) * V, c->beta[(long)b * HV + hv],
                      c->a + ((long)b * HV + hv) * K, c->o + ((long)b * HV + hv) * V, NULL);
    }
}

/* One KDA decode step over the batch; a is [batch][HV][K]. */
int orc_kda_step(const orc_gdn_dims* d, double* state, const double* q, const double* k,
                 const double* v, const double* beta, const double* a, const int* ci,
                 double* o, int nthreads) {
    if (d->num_k_heads <= 0 || d->num_v_heads % d->num_k_heads) return 3;
    kda_step_ctx c = {d, state, q, k, v, beta, a, ci, o};
    for_rows(kda_step_row, &c, d->batch, nthreads);
    return 0;
}

typedef struct {
    const orc_gdn_dims* d;
    int L;
    const double* S0;
    const int *ci, *wp;
    const double *ek, *ev, *ebeta, *ea, *q;
    double *o, *S_fold, *d_out;
} kda_replay_ctx;

/* ReplaySSM closed form of the KDA step (checkpoint S0 + ring of (d, k, a)):
 * with D_i = Diag(a_i) and S^(i) = S^(i-1) D_i + d_i k_i^T, S^(-1) = S0,
 *   S^(i-1) D_i k_i = S0 (prod_{j<=i} D_j) k_i
 *                   + sum_{m<i} d_m k_m^T (prod_{j=m+1..i} D_j) k_i
 *   d_i = beta_i (v_i - S^(i-1) D_i k_i)
 *   o_w = S0 (prod_{j<=w} D_j) q + sum_{m<=w} d_m k_m^T (prod_{j=m+1..w} D_j) q
 *   S^(w) = S0 prod_{j<=w} D_j + sum_{m<=w} d_m k_m^T prod_{j=m+1..w} D_j  (flush)
 * where every product of diagonal gates is a per-channel product. Entry arrays
 * per row: ek[b][i][HK][K], ev[b][i][HV][V], ebeta[b][i][HV], ea[b][i][HV][K];
 * q is the current q[b][HK][K]. Outputs as orc_gdn_replay. */
static void kda_replay_row(const void* vctx, int b) {
    const kda_replay_ctx* c = (const kda_replay_ctx*)vctx;
    const orc_gdn_dims* d = c->d;
    const int HV = d->num_v_heads, HK = d->num_k_heads, K = d->head_k_dim, V = d->head_v_dim;
    const int L = c->L;
    const int s = c->ci[b];
    if (s < 0 || s >= d->num_slots) return;
    const int w = c->wp[b];
    const int vpk = HV / HK;
    double* dd = (double*)malloc(sizeof(double) * (long)(w + 1) * V);
    double* tmp = (double*)malloc(sizeof(double) * V);
    double* gam = (double*)malloc(sizeof(double) * K);
    for (int hv = 0; hv < HV; ++hv) {
        const int kh = hv / vpk;
        const double* S0 = c->S0 + (((long)s * HV + hv) * V) * K;
#define KDA_A(i, ik) c->ea[(((long)b * L + (i)) * HV + hv) * K + (ik)]
#define KDA_K(i, ik) c->ek[(((long)b * L + (i)) * HK + kh) * K + (ik)]
        for (int i = 0; i <= w; ++i) {
            /* S0 term: gam = prod_{j<=i} a_j */
            for (int ik = 0; ik < K; ++ik) {
                double g = 1.0;
                for (int j = 0; j <= i; ++j) g *= KDA_A(j, ik);
                gam[ik] = g;
            }
            for (int iv = 0; iv < V; ++iv) {
                double acc = 0.0;
                for (int ik = 0; ik < K; ++ik) acc += S0[(long)iv * K + ik] * gam[ik] * KDA_K(i, ik);
                tmp[iv] = acc;
            }
            for (int m = 0; m < i; ++m) {
                double kk = 0.0;
                for (int ik = 0; ik < K; ++ik) {
                    double g = 1.0;
                    for (int j = m + 1; j <= i; ++j) g *= KDA_A(j, ik);
                    kk += KDA_K(m, ik) * g * KDA_K(i, ik);
                }
                for (int iv = 0; iv < V; ++iv) tmp[iv] += dd[(long)m * V + iv] * kk;
            }
            const double be = c->ebeta[((long)b * L + i) * HV + hv];
            const double* vi = c->ev + (((long)b * L + i) * HV + hv) * V;
            for (int iv = 0; iv < V; ++iv) dd[(long)i * V + iv] = be * (vi[iv] - tmp[iv]);
        }
        const double* q = c->q + ((long)b * HK + kh) * K;
        for (int ik = 0; ik < K; ++ik) {
            double g = 1.0;
            for (int j = 0; j <= w; ++j) g *= KDA_A(j, ik);
            gam[ik] = g;
        }
        for (int iv = 0; iv < V; ++iv) {
            double acc = 0.0;
            for (int ik = 0; ik < K; ++ik) acc += S0[(long)iv * K + ik] * gam[ik] * q[ik];
            tmp[iv] = acc;
        }
        for (int m = 0; m <= w; ++m) {
            double kq = 0.0;
            for (int ik = 0; ik < K; ++ik) {
                double g = 1.0;
                for (int j = m + 1; j <= w; ++j) g *= KDA_A(j, ik);
                kq += KDA_K(m, ik) * g * q[ik];
            }
            for (int iv = 0; iv < V; ++iv) tmp[iv] += dd[(long)m * V + iv] * kq;
        }
        for (int iv = 0; iv < V; ++iv) c->o[((long)b * HV + hv) * V + iv] = tmp[iv];
        if (c->d_out)
            for (int i = 0; i <= w; ++i)
                for (int iv = 0; iv < V; ++iv)
                    c->d_out[(((long)b * L + i) * HV + hv) * V + iv] = dd[(long)i * V + iv];
        if (c->S_fold) {
            double* Sf = c->S_fold + (((long)b * HV + hv) * V) * K;
            for (int iv = 0; iv < V; ++iv)
                for (int ik = 0; ik < K; ++ik) {
                    double val = S0[(long)iv * K + ik] * gam[ik];
                    for (int m = 0; m <= w; ++m) {
                        double g = 1.0;
                        for (int j = m + 1; j <= w; ++j) g *= KDA_A(j, ik);
                        val += dd[(long)m * V + iv] * KDA_K(m, ik) * g;
                    }
                    Sf[(long)iv * K + ik] = val;
                }
        }
#undef KDA_A
#undef KDA_K
    }
    free(dd); free(tmp); free(gam);
}

int orc_kda_replay(const orc_gdn_dims* d, int L, const double* S0, const int* ci, const int* wp,
                   const double* ek, const double* ev, const double* ebeta, const double* ea,
                   const double* q, double* o, double* S_fold, double* d_out, int nthreads) {
    if (d->num_k_heads <= 0 || d->num_v_heads % d->num_k_heads) return 3;
    for (int b = 0; b < d->batch; ++b)
        if (ci[b] >= 0 && (wp[b] < 0 || wp[b] >= L)) return 1;
    kda_replay_ctx c = {d, L, S0, ci, wp, ek, ev, ebeta, ea, q, o, S_fold, d_out};
    for_rows(kda_replay_row, &c, d->batch, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Gated delta net: one speculative verify round                             */
/* ------------------------------------------------------------------------- */

typedef struct {
    const orc_gdn_dims* d;
    int T;
    double* state;
    const double *q, *k, *v, *beta, *g;
    const int *ci, *acc;
    double* o;
} gdn_spec_ctx;

/* [SPEC] 实现拆解 items 3-4: a verify round scores a linear chain of T draft
 * tokens. Draft j's output is the recurrence output after the committed history
 * and drafts 0..j (rejected drafts included). The commit then keeps the state
 * after the first acc[b] drafts only (acc in 0..T); the rest are discarded.
 * Inputs per row and draft: q,k [b][T][HK][K], v [b][T][HV][V], beta,g [b][T][HV].
 * o receives [b][T][HV][V]. Each head is run on a private copy of its state. */
static void gdn_spec_row(const void* vctx, int b) {
    const gdn_spec_ctx* c = (const gdn_spec_ctx*)vctx;
    const orc_gdn_dims* d = c->d;
    const int HV = d->num_v_heads, HK = d->num_k_heads, K = d->head_k_dim, V = d->head_v_dim;
    const int T = c->T;
    const int s = c->ci[b];
    if (s < 0 || s >= d->num_slots) return;
    const int acc = c->acc[b];
    const int vpk = HV / HK;
    double* S = (double*)malloc(sizeof(double) * (long)V * K);
    for (int hv = 0; hv < HV; ++hv) {
        const int kh = hv / vpk;
        double* Sslot = c->state + (((long)s * HV + hv) * V) * K;
        memcpy(S, Sslot, sizeof(double) * (long)V * K);
        for (int j = 0; j < T; ++j) {
            const long bj = (long)b * T + j;
            gdn_head_step(S, K, V, c->q + (bj * HK + kh) * K, c->k + (bj * HK + kh) * K,
                          c->v + (bj * HV + hv) * V, c->beta[bj * HV + hv], c->g[bj * HV + hv],
                          c->o + (bj * HV + hv) * V, NULL);
            if (j + 1 == acc) memcpy(Sslot, S, sizeof(double) * (long)V * K);
        }
    }
    free(S);
}

int orc_gdn_spec_round(const orc_gdn_dims* d, int T, double* state, const double* q,
                       const double* k, const double* v, const double* beta, const double* g,
                       const int* ci, const int* acc, double* o, int nthreads) {
    if (d->num_k_heads <= 0 || d->num_v_heads % d->num_k_heads) return 3;
    for (int b = 0; b < d->batch; ++b)
        if (ci[b] >= 0 && (acc[b] < 0 || acc[b] > T)) return 1;
    gdn_spec_ctx c = {d, T, state, q, k, v, beta, g, ci, acc, o};
    for_rows(gdn_spec_row, &c, d->batch, nthreads);
    return 0;
}
