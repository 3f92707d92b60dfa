/*
 * rssm.h -- C ABI of librssm.so: ReplaySSM decode for Mamba2 and gated delta net
 * on GB300 (sm_103a).
 *
 * ReplaySSM keeps, per state slot, a frozen checkpoint S0 of the recurrent state
 * plus a ring of the last L steps' inputs. A decode step computes its output from
 * S0 and the ring instead of reading and writing the whole state; the state is
 * folded and written back only on flush rows (every L steps, or when forced).
 *
 * Pages this interface follows (cited by title and section):
 *   [M2]   "ReplaySSM: cache SSM inputs for faster Mamba2 standard decode"
 *          (vLLM PR 48018 report): 功能与动机 (motivation), 实现拆解 items 1-3
 *          (precompute + output kernels, ring append, per-row write_pos/is_flush
 *          from the metadata builder), 关键源码片段 (the kernel call with
 *          ssm_state, x, dt, A, B, C, D, x_cache, dt_cache, B_cache, write_pos,
 *          is_flush, state_batch_indices, out, dt_bias, dt_softplus), 评论区精华
 *          (stochastic rounding of the state), 关联脉络 (the full design also
 *          covers speculative decode).
 *   [FI]   "[Mamba] Add FlashInfer ReplaySSM backend" (vLLM PR 52506 report):
 *          实现拆解 items 1-2 (ring cursor update/reset kernels; one cursor
 *          advance shared by all layers of a cache group).
 *   [GDN]  "GDN ReplaySSM decode (Part A of RFC 28511)" (SGLang PR 28451 report):
 *          实现拆解 items 1-3 (decode kernel over the (d, k, g) ring, flush every L
 *          steps, CUDA-graph-safe write_pos and force-flush buffers; the KDA
 *          per-K gate; copy_from with the rings), 评论区精华 (KDA gate ring).
 *   [SPEC] "[GDN] Support ReplaySSM Ring Spec-Verify" (SGLang PR 28695 report):
 *          实现拆解 items 2-4 (circular ring, cursors write_pos / cache_base /
 *          is_flush, spec verify kernel, exact fold from raw inputs, commit that
 *          only advances cursors), 关键源码片段 (ring length >= 2 x drafts).
 *
 * Conventions for every entry point:
 *   - Every pointer argument is a DEVICE pointer owned by the caller, 16-byte
 *     aligned, to a dense row-major array with the layout stated below. The
 *     library allocates nothing and keeps no reference after the call returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). No call synchronises or reads device data on the host, so
 *     every call may be captured in a CUDA graph.
 *   - Arguments are validated on the host before anything is launched; a call
 *     that returns an error has launched nothing and changed nothing.
 *   - Return value: RSSM_OK, or an RSSM_ERR_* code (rssm_status_string()).
 *   - Device-detected problems cannot be returned synchronously. Where a call
 *     takes `int32_t* dev_err` (nullable), a kernel that finds a row with a cache
 *     index >= num_slots, or a cursor outside [0, L), skips that row and ORs an
 *     RSSM_DEVERR_* bit into *dev_err. Rows whose cache index is negative are
 *     padding (as in padded CUDA-graph batches): they are skipped silently and
 *     their outputs are left untouched.
 *   - Two rows of one call must not name the same slot (undefined result).
 *   - Shapes named: b = batch row, s = slot = cache_indices[b], H = nheads,
 *     P = headdim, N = dstate, G = ngroups, L = ring length; for the gated delta
 *     net HV = value heads, HK = key heads, K = key dim, V = value dim.
 *
 * Storage dtypes: RSSM_F32 (IEEE float32) or RSSM_BF16 (bfloat16). State stores
 * round to nearest, ties to even, except through the *_sr entry points (stochastic
 * rounding of a bf16 Mamba2 state). All arithmetic accumulates in float32.
 */
#ifndef RSSM_H
#define RSSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* rssm_stream_t;

#define RSSM_ABI_VERSION 1

enum rssm_status {
    RSSM_OK = 0,
    RSSM_ERR_INVALID_ARG = 1, /* null or misaligned pointer, bad enum, negative size */
    RSSM_ERR_UNSUPPORTED = 2, /* shape or dtype this build has no kernel for */
    RSSM_ERR_CONFIG = 3,      /* inconsistent configuration (nheads % ngroups, L < 1, L < 2T ...) */
    RSSM_ERR_CUDA = 4         /* the CUDA runtime reported an error at launch */
};

enum rssm_dtype { RSSM_F32 = 0, RSSM_BF16 = 1 };

/* Bits ORed into *dev_err by kernels. */
enum rssm_dev_error {
    RSSM_DEVERR_SLOT = 1,    /* a row's cache index was >= num_slots; the row was skipped */
    RSSM_DEVERR_CURSOR = 2,  /* a row's write_pos / count was outside the ring; row skipped */
    RSSM_DEVERR_TIMEOUT = 4  /* a bounded wait on an asynchronous copy expired; kernel stopped */
};

/* Cursor modes of rssm_advance_cursors. */
enum rssm_cursor_mode {
    RSSM_CURSOR_STANDARD = 0,
    RSSM_CURSOR_SPEC_COMMIT = 1,
    RSSM_CURSOR_RESET = 2
};

/* Text for a status code (static storage; never NULL). */
const char* rssm_status_string(int status);

/* RSSM_ABI_VERSION of the loaded library. */
int rssm_abi_version(void);

/* ------------------------------------------------------------------------- */
/* Cursors                                                                    */
/* ------------------------------------------------------------------------- */

/* rssm_advance_cursors -- per-row ring cursors, computed on the device so that a
 * captured decode step needs no host metadata. One launch serves every layer
 * that shares the slots ([FI] 实现拆解 item 2: one tracker advance per cache
 * group; [M2] 实现拆解 item 3: write_pos / is_flush per decode row).
 *
 * RSSM_CURSOR_STANDARD ([M2], [GDN] 实现拆解 item 2). For each row b with
 *   s = cache_indices[b] >= 0:  w = slot_wp[s];
 *   f = (w == L-1) || (force_flush && force_flush[b]);
 *   row_wp[b] = w; row_flush[b] = f; slot_wp[s] = f ? 0 : w + 1.
 *   Padding rows get row_wp = 0, row_flush = 0. Entry w of the ring is the
 *   current step; a flush folds entries 0..w into the checkpoint.
 *   Uses slot_wp [num_slots], cache_indices [batch], force_flush [batch]
 *   (nullable), row_wp [batch], row_flush [batch]. slot_base, slot_flush,
 *   num_accepted, T unused (may be NULL / 0).
 *
 * RSSM_CURSOR_SPEC_COMMIT ([SPEC] 实现拆解 item 4: the commit only advances
 *   cursors). Per slot: slot_wp = committed unfolded entry count cnt, slot_base =
 *   ring position of the oldest unfolded entry, slot_flush = fold pending. For
 *   each row with s >= 0:
 *     if slot_flush[s]: slot_base[s] = (slot_base[s] + slot_wp[s]) % L; slot_wp[s] = 0;
 *     slot_wp[s] += num_accepted[b];   (0 <= num_accepted[b] <= T)
 *     slot_flush[s] = (slot_wp[s] + T > L);
 *   and, when given, row_wp[b] / row_flush[b] receive the new cnt / flush.
 *   Must follow the rssm_gdn_spec_verify call of the same round.
 *
 * RSSM_CURSOR_RESET ([FI] reset_replayssm_ring_trackers; [SPEC] cursor reset at
 *   slot (re)use): for each row with s >= 0, slot_wp[s] = 0 and, when given,
 *   slot_base[s] = 0, slot_flush[s] = 0.
 *
 * Errors: RSSM_ERR_INVALID_ARG for a NULL required pointer; RSSM_ERR_CONFIG for
 * L < 1, or, in SPEC_COMMIT, T < 1 or L < 2T. A num_accepted outside [0, T] or a
 * stored cursor outside the ring sets RSSM_DEVERR_CURSOR and leaves that slot. */
int rssm_advance_cursors(int mode, int32_t* slot_wp, int32_t* slot_base, uint8_t* slot_flush,
                         const int32_t* cache_indices, const uint8_t* force_flush,
                         const int32_t* num_accepted, int32_t batch, int32_t num_slots,
                         int32_t L, int32_t T, int32_t* row_wp, uint8_t* row_flush,
                         int32_t* dev_err, rssm_stream_t stream);

/* Slot fork ("GDN ReplaySSM decode (Part A of RFC 28511)", 实现拆解 item 3: the
 * memory pool's copy_from copies the ring buffers with the state and sets the
 * cursors; 评论区精华: copying a slot whose ring still holds live entries must not
 * lose them).
 *
 * A slot-indexed buffer: slot s occupies bytes [base + s * slot_bytes, base + (s+1)
 * * slot_bytes) of a device array. */
typedef struct rssm_slot_buffer {
    void* base;        /* device pointer (16-byte aligned base and size copy fastest) */
    size_t slot_bytes; /* bytes per slot, > 0 */
} rssm_slot_buffer;

#define RSSM_MAX_SLOT_BUFFERS 12

/* rssm_copy_slots -- for i < n: copy slot src_slots[i]'s record into slot
 * dst_slots[i] in every listed buffer. List every per-slot buffer of the cache --
 * checkpoint, rings and cursors (Mamba2: state, ring_x, ring_dt, ring_B, slot_wp;
 * gated delta net: state, ring_d, ring_k, ring_g, slot_wp; spec adds ring_v,
 * ring_beta, slot_base, slot_flush) -- and the destination continues exactly as
 * the source would (live ring entries and the cursor position are carried, so the
 * source need not have flushed).
 *   buffers: HOST array of n_buffers (1 .. RSSM_MAX_SLOT_BUFFERS) descriptors;
 *     read during the call only.
 *   src_slots, dst_slots: device int32 [n]. A pair with a negative entry is
 *     skipped (padding); an entry >= num_slots skips the pair and sets
 *     RSSM_DEVERR_SLOT; src == dst is a no-op. Destinations must be distinct and
 *     must not be sources of the same call (undefined result otherwise).
 * Errors: RSSM_ERR_INVALID_ARG for a NULL buffers array or base, n_buffers outside
 * 1..RSSM_MAX_SLOT_BUFFERS, slot_bytes == 0, n < 0, num_slots <= 0, or (n > 0)
 * NULL / misaligned slot arrays. */
int rssm_copy_slots(const rssm_slot_buffer* buffers, int32_t n_buffers, const int32_t* src_slots,
                    const int32_t* dst_slots, int32_t n, int32_t num_slots, int32_t* dev_err,
                    rssm_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Mamba2                                                                     */
/* ------------------------------------------------------------------------- */

typedef struct rssm_mamba2_dims {
    int32_t batch;       /* rows in this call (>= 0) */
    int32_t nheads;      /* H */
    int32_t headdim;     /* P: 64 or 128 */
    int32_t dstate;      /* N: 64 or 128 */
    int32_t ngroups;     /* G: H % G == 0; heads h*G/H .. share group h / (H/G) */
    int32_t ring_len;    /* L >= 1 */
    int32_t num_slots;   /* slots in the state pool and the rings */
    int32_t state_dtype; /* RSSM_F32 | RSSM_BF16: state pool */
    int32_t act_dtype;   /* RSSM_F32 | RSSM_BF16: x, z, B, C, ring_x, ring_B */
    int32_t out_dtype;   /* RSSM_F32 | RSSM_BF16: y */
} rssm_mamba2_dims;

/* Layouts (row-major, dense):
 *   state   [num_slots][H][P][N]  state_dtype   checkpoint S0 per slot
 *   ring_x  [num_slots][H][L][P]  act_dtype     x of each ring entry
 *   ring_dt [num_slots][H][L]     float32       dt = softplus(dt_raw + dt_bias) per entry
 *   ring_B  [num_slots][G][L][N]  act_dtype     B of each ring entry
 *   x, z    [batch][H][P]         act_dtype
 *   dt_raw  [batch][H]            float32
 *   B, C    [batch][G][N]         act_dtype
 *   A, D, dt_bias [H]             float32
 *   y       [batch][H][P]         out_dtype
 *   cache_indices [batch] int32; row_wp [batch] int32; row_flush [batch] uint8
 *   (as produced by rssm_advance_cursors STANDARD). */

/* rssm_ring_append -- write the current step's (x, dt, B) into ring entry
 * row_wp[b] of slot cache_indices[b] ([M2] 关键符号 append_replayssm_ring;
 * 实现拆解 item 2: x_cache, dt_cache, B_cache). The stored dt is
 * softplus(dt_raw + dt_bias[h]) when dt_softplus is non-zero, else
 * dt_raw + dt_bias[h]; dt_bias may be NULL (zero). Heads of one group write the
 * group's B once. */
int rssm_ring_append(const rssm_mamba2_dims* dims, const void* x, const float* dt_raw,
                     const float* dt_bias, int dt_softplus, const void* B,
                     const int32_t* cache_indices, const int32_t* row_wp, void* ring_x,
                     float* ring_dt, void* ring_B, int32_t* dev_err, rssm_stream_t stream);

/* Bytes of device workspace rssm_mamba2_precompute / rssm_mamba2_decode need: the
 * per-(row, head) coefficient tables, float32 (batch * nheads * round4(2L + 1) * 4
 * bytes), then, at the next 256-byte boundary, 256 bytes for the output kernel's work
 * counter (the table-building launches zero it every step; the output launch claims
 * its tiles from it and leaves it at zero). A workspace serves one stream at a time.
 * 0 for an invalid dims. */
size_t rssm_mamba2_workspace_size(const rssm_mamba2_dims* dims);

/* rssm_mamba2_precompute -- per-row scalar tables for the output kernel ([M2]
 * 实现拆解 item 1: the precompute kernel). For row b, head h, entries i = 0..w
 * (w = row_wp[b]), with dA_j = exp(A[h] * dt_j) and dt_j read from ring_dt:
 *   P_i  = prod_{j=i+1..w} dA_j  (= exp(A[h] * sum_{j>i} dt_j)),
 *   Pm1  = prod_{j=0..w} dA_j,
 *   bc_i = B_i . C_t over dstate (B_i from ring_B, group of h),
 *   coef_i = P_i dt_i bc_i, a_i = P_i dt_i;
 * stored per (b, h) as [coef_0..coef_{L-1}, a_0..a_{L-1}, Pm1, pad] in workspace.
 * The ring must already hold the current entry (rssm_ring_append). */
int rssm_mamba2_precompute(const rssm_mamba2_dims* dims, const float* A, const void* C,
                           const float* ring_dt, const void* ring_B,
                           const int32_t* cache_indices, const int32_t* row_wp,
                           void* workspace, size_t workspace_bytes, int32_t* dev_err,
                           rssm_stream_t stream);

/* rssm_mamba2_output -- the fused output / flush kernel ([M2] 实现拆解 item 1:
 * output kernel branching per row on is_flush; 功能与动机: most steps read the
 * output from checkpoint + buffer, the full state is written back every L
 * steps). Streams each (row, head) checkpoint tile S0 once:
 *   y[p] = Pm1 * sum_n S0[p][n] C[n] + sum_{i=0..w} coef_i x_i[p] + D[h] x_w[p],
 *   y[p] *= silu(z[p])   (z nullable)
 * and, on flush rows, stores state[s][h] = Pm1 * S0 + sum_i a_i x_i B_i^T
 * rounded to state_dtype. Needs the tables of rssm_mamba2_precompute. */
int rssm_mamba2_output(const rssm_mamba2_dims* dims, void* state, const void* C, const float* D,
                       const void* z, const void* ring_x, const void* ring_B,
                       const int32_t* cache_indices, const int32_t* row_wp,
                       const uint8_t* row_flush, const void* workspace, size_t workspace_bytes,
                       void* y, int32_t* dev_err, rssm_stream_t stream);

/* rssm_mamba2_decode -- rssm_mamba2_precompute then rssm_mamba2_output (the
 * selective_state_update_replayssm_output_only call of [M2] 关键源码片段). */
int rssm_mamba2_decode(const rssm_mamba2_dims* dims, void* state, const float* A, const void* C,
                       const float* D, const void* z, const void* ring_x, const float* ring_dt,
                       const void* ring_B, const int32_t* cache_indices, const int32_t* row_wp,
                       const uint8_t* row_flush, void* workspace, size_t workspace_bytes,
                       void* y, int32_t* dev_err, rssm_stream_t stream);

/* rssm_mamba2_prepare -- the per-row prologue of one decode step in ONE launch
 * (one CTA per row): the STANDARD cursor step of rssm_advance_cursors (when
 * advance != 0), rssm_ring_append, then rssm_mamba2_precompute. Results are
 * those of the three calls in that order ([M2] 实现拆解 items 1 and 3: the
 * per-row precompute runs before the output kernel, write_pos / is_flush per
 * row). With advance == 0 the row cursors come from an earlier
 * rssm_advance_cursors (layers that share one advance); slot_wp, force_flush and
 * row_flush are then unused (may be NULL). Arguments and layouts as in those
 * calls; errors as theirs. */
int rssm_mamba2_prepare(const rssm_mamba2_dims* dims, int advance, const uint8_t* force_flush,
                        int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush, const void* x,
                        const float* dt_raw, const float* dt_bias, int dt_softplus,
                        const void* B, const float* A, const void* C,
                        const int32_t* cache_indices, void* ring_x, float* ring_dt,
                        void* ring_B, void* workspace, size_t workspace_bytes,
                        int32_t* dev_err, rssm_stream_t stream);

/* rssm_mamba2_step -- one whole ReplaySSM decode step in two launches:
 * rssm_mamba2_prepare then rssm_mamba2_output ([M2] 关键源码片段: the decode
 * path calls the ReplaySSM update once per step in place of
 * selective_state_update). row_flush is always required (the output kernel reads
 * it). Arguments, layouts and errors as in those two calls.
 * Small batches (batch <= 16, advance = 1, ring_len <= 64) take one launch
 * instead ([M2] 风险与影响 item 3: at batch 1-8 the step is bound by launch
 * latency): a CTA per (row, head) advances the cursor, appends the row's entry,
 * builds its head's table and computes y and the fold, with identical results up
 * to float32 rounding order (the tables are not left in the workspace). The last
 * CTA of a row advances the slot cursor through a per-row counter in the
 * workspace's 256-byte counter block (rssm_mamba2_workspace_size), so the
 * workspace must be zero-filled before its first use with this call; the call
 * leaves those counters at zero. */
int rssm_mamba2_step(const rssm_mamba2_dims* dims, int advance, const uint8_t* force_flush,
                     int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush, void* state,
                     const void* x, const float* dt_raw, const float* dt_bias, int dt_softplus,
                     const float* A, const void* B, const void* C, const float* D, const void* z,
                     const int32_t* cache_indices, void* ring_x, float* ring_dt, void* ring_B,
                     void* workspace, size_t workspace_bytes, void* y, int32_t* dev_err,
                     rssm_stream_t stream);

/* Stochastic rounding of the bf16 state store ([M2] 评论区精华: quantised models
 * such as the NVFP4 Nemotron baseline rely on stochastic rounding of the state,
 * and the report adds it as an option).
 *
 * sr_state is a DEVICE array of two uint64: {seed, offset}. A state element with
 * float32 value f at element index e of the state pool (e = ((s * H + h) * P + p)
 * * N + n) is stored as the bf16 obtained by adding r_e (16 random bits) to the
 * bit pattern of f and dropping the low 16 bits, so it rounds up with probability
 * equal to the dropped fraction (unbiased); NaN and +-Inf are stored as with
 * round-to-nearest. The bits come from Philox4x32-10 (Salmon, Moraes, Dror and
 * Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011) with key = seed
 * (low word first) and counter = {e / 8 low, e / 8 high, offset low, offset high}:
 * its four 32-bit outputs w0..w3 give r for the 8 elements e0 = 8 (e / 8) + j as
 * the low (j even) or high (j odd) half of w_{j / 2}. After every launch that
 * stores a state, the call adds 1 to offset (on the device, in stream order), so
 * graph replays draw fresh bits. For a float32 state the generator is not used
 * (offset still advances). sr_state must not be NULL; errors as in the call
 * without _sr. */

/* rssm_mamba2_output with stochastic rounding of the flush stores (see above). */
int rssm_mamba2_output_sr(const rssm_mamba2_dims* dims, void* state, const void* C,
                          const float* D, const void* z, const void* ring_x, const void* ring_B,
                          const int32_t* cache_indices, const int32_t* row_wp,
                          const uint8_t* row_flush, const void* workspace,
                          size_t workspace_bytes, void* y, uint64_t* sr_state, int32_t* dev_err,
                          rssm_stream_t stream);

/* rssm_mamba2_step with stochastic rounding of the flush stores (see above). */
int rssm_mamba2_step_sr(const rssm_mamba2_dims* dims, int advance, const uint8_t* force_flush,
                        int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush, void* state,
                        const void* x, const float* dt_raw, const float* dt_bias,
                        int dt_softplus, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const int32_t* cache_indices,
                        void* ring_x, float* ring_dt, void* ring_B, void* workspace,
                        size_t workspace_bytes, void* y, uint64_t* sr_state, int32_t* dev_err,
                        rssm_stream_t stream);

/* rssm_philox4x32_fill -- out[4 g .. 4 g + 3] = Philox4x32-10(counter {g low,
 * g high, offset low, offset high}, key {seed low, seed high}) for g < n_groups:
 * the bits the stochastic rounding of 8-element group g draws at that offset (a
 * debug / test entry point). out: device uint32 [4 n_groups]. */
int rssm_philox4x32_fill(uint64_t seed, uint64_t offset, uint32_t* out, size_t n_groups,
                         rssm_stream_t stream);

/* Bytes of workspace rssm_mamba2_spec_verify needs for T drafts (per-(row, head)
 * tables: T x L coefficients, T decay products, T draft dt). 0 for invalid dims
 * or T outside 1..4. */
size_t rssm_mamba2_spec_workspace_size(const rssm_mamba2_dims* dims, int32_t T);

/* rssm_mamba2_spec_verify -- score T draft tokens per row from the checkpoint and
 * the circular ring, without per-draft states ([M2] 关联脉络: the full ReplaySSM
 * design covers Mamba2 speculative decode; the ring, cursors, fold and commit
 * follow [SPEC] 实现拆解 items 2-4, as for rssm_gdn_spec_verify). Two launches: a
 * prologue that folds, for slots whose fold is pending (slot_flush), the committed
 * entries into the checkpoint (S0 <- prod dA_i S0 + sum_i (prod_{l>i} dA_l) dt_i
 * x_i B_i^T, rounded to state_dtype) and builds the draft tables; then the verify,
 * which reads each checkpoint tile once for all drafts:
 *   y_j = (prod_{i<=m} dA_i) S0 C_j + sum_{i<=m} (prod_{l=i+1..m} dA_l) dt_i (B_i . C_j) x_i
 *         + D x_j,  gated by silu(z_j),  m = history + j,
 * over the history entries (ring positions (base + i) % L, i < cnt) and drafts
 * 0..j, and writes draft j's x, dt (after softplus) and B at ring position
 * (base + cnt + j) % L. Commit with rssm_advance_cursors(RSSM_CURSOR_SPEC_COMMIT).
 * Cursors (read only here): slot_cnt = cnt, slot_base = base, slot_flush = fold
 * pending (the ring length must hold twice the drafts).
 * Inputs per draft: x, z [batch][T][H][P] (z nullable), dt_raw [batch][T][H]
 * float32, B, C [batch][T][G][N] (act_dtype); A, D, dt_bias as in decode. Ring
 * layouts as in decode. Output y [batch][T][H][P] (out_dtype).
 * Errors: RSSM_ERR_UNSUPPORTED for T outside 1..4 or L > 32; RSSM_ERR_CONFIG for L < 2T; a
 * slot whose cursors break cnt + T <= L (without a pending fold) is skipped and
 * flagged RSSM_DEVERR_CURSOR. */
int rssm_mamba2_spec_verify(const rssm_mamba2_dims* dims, int32_t T, void* state, const void* x,
                            const float* dt_raw, const float* dt_bias, int dt_softplus,
                            const float* A, const void* B, const void* C, const float* D,
                            const void* z, void* ring_x, float* ring_dt, void* ring_B,
                            const int32_t* cache_indices, const int32_t* slot_cnt,
                            const int32_t* slot_base, const uint8_t* slot_flush, void* workspace,
                            size_t workspace_bytes, void* y, int32_t* dev_err,
                            rssm_stream_t stream);

/* Size of the device array rssm_mamba2_decode_noalloc keeps its workspace in. */
#define RSSM_NOALLOC_WORKSPACE_BYTES (16u << 20)

/* rssm_mamba2_decode_noalloc -- rssm_mamba2_decode for callers that cannot allocate
 * device memory. The pages have no counterpart: this is an interface for such
 * callers, not part of the method. Some callers cannot provide the workspace that
 * rssm_mamba2_decode needs -- a plug-in inside a host application that owns every
 * device allocation, an engine whose device memory budget is fixed at start-up, a
 * caller on a latency-critical path that must never enter the allocator. This
 * entry point takes the same inputs and outputs (all device pointers, caller
 * owned) but no workspace: the coefficient tables live in a fixed array of
 * RSSM_NOALLOC_WORKSPACE_BYTES (16 MiB) inside the library's device image, held
 * by every GPU that loads the library until the process exits. It allocates
 * nothing and calls no allocating routine.
 *   - Limit: rssm_mamba2_workspace_size(dims) must not exceed the array (the
 *     tables, batch * nheads * round4(2L + 1) * 4 bytes, plus 256 bytes rounded;
 *     batch 512 x 128 heads at L = 16 needs 9 MiB); larger sizes return
 *     RSSM_ERR_UNSUPPORTED before any launch.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call before
 *     any stream capture. A failed look-up returns RSSM_ERR_CUDA and is not cached:
 *     the next call tries again. The address is kept per device together with the
 *     id of the context it belongs to; after cudaDeviceReset (a new context, the
 *     module loaded again) the next call looks it up again, so that call too should
 *     come before any stream capture.
 *   - Sharing: every call on a device uses the same array and leaves its contents
 *     there; nothing in it needs to start at zero. Calls whose executions overlap on
 *     the GPU race on it, so keep them in one stream or order them.
 * Other arguments, results and errors are those of rssm_mamba2_decode. */
int rssm_mamba2_decode_noalloc(const rssm_mamba2_dims* dims, void* state, const float* A,
                               const void* C, const float* D, const void* z, const void* ring_x,
                               const float* ring_dt, const void* ring_B,
                               const int32_t* cache_indices, const int32_t* row_wp,
                               const uint8_t* row_flush, void* y, int32_t* dev_err,
                               rssm_stream_t stream);

/* rssm_mamba2_full_state_update -- the conventional decode step that reads and
 * writes the whole state every step ([M2] 关键源码片段, the baseline
 * selective_state_update branch). For each row with s >= 0, head h:
 *   dt = softplus(dt_raw + dt_bias) (or without softplus), dA = exp(A[h] dt),
 *   h = dA h + dt x B^T (stored rounded to state_dtype),
 *   y = (h C + D x) * silu(z)  (from the unrounded h; z nullable).
 * ring_len is ignored. */
int rssm_mamba2_full_state_update(const rssm_mamba2_dims* dims, void* state, const void* x,
                                  const float* dt_raw, const float* dt_bias, int dt_softplus,
                                  const float* A, const void* B, const void* C, const float* D,
                                  const void* z, const int32_t* cache_indices, void* y,
                                  int32_t* dev_err, rssm_stream_t stream);

/* rssm_mamba2_full_state_update with stochastic rounding of the state store
 * (the rounding of rssm_mamba2_output_sr). */
int rssm_mamba2_full_state_update_sr(const rssm_mamba2_dims* dims, void* state, const void* x,
                                     const float* dt_raw, const float* dt_bias, int dt_softplus,
                                     const float* A, const void* B, const void* C,
                                     const float* D, const void* z,
                                     const int32_t* cache_indices, void* y, uint64_t* sr_state,
                                     int32_t* dev_err, rssm_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Gated delta net                                                            */
/* ------------------------------------------------------------------------- */

typedef struct rssm_gdn_dims {
    int32_t batch;       /* rows in this call (>= 0) */
    int32_t num_v_heads; /* HV */
    int32_t num_k_heads; /* HK: HV % HK == 0; value head hv reads key head hv / (HV/HK) */
    int32_t head_k_dim;  /* K: 128 */
    int32_t head_v_dim;  /* V: multiple of 32 */
    int32_t ring_len;    /* L >= 1 */
    int32_t num_slots;
    int32_t act_dtype;   /* RSSM_F32 | RSSM_BF16: q, k, v, ring_k, ring_v */
    int32_t out_dtype;   /* RSSM_F32 | RSSM_BF16: o */
} rssm_gdn_dims;

/* Layouts (row-major, dense); the state is float32 ([SPEC] 风险与影响: the
 * ReplaySSM path keeps an fp32 checkpoint):
 *   state   [num_slots][HV][V][K] float32  checkpoint S0 per slot
 *   ring_d  [num_slots][HV][V/32][L][32] float32  d_i = beta_i (v_i - g_i S_{i-1} k_i),
 *           value rows in blocks of 32 (one block's L entries are contiguous)
 *   ring_k  [num_slots][HK][L][K] act_dtype
 *   ring_g  [num_slots][HV][L]    float32  gate value g_i in (0, 1]
 *   q, k    [batch][HK][K] act_dtype; v [batch][HV][V] act_dtype
 *   beta, g [batch][HV] float32; o [batch][HV][V] out_dtype
 * The recurrence is S <- g S + beta (v - g S k) k^T, o = S q ([GDN] 功能与动机:
 * the conventional kernel reads and writes S[HV, V, K] every step). */

/* rssm_gdn_ring_append -- write k and g of the current step into ring entry
 * row_wp[b] ([GDN] 实现拆解 item 1, the (d, k, g) ring). d is produced by the
 * output kernel, which needs the state. */
int rssm_gdn_ring_append(const rssm_gdn_dims* dims, const void* k, const float* g,
                         const int32_t* cache_indices, const int32_t* row_wp, void* ring_k,
                         float* ring_g, int32_t* dev_err, rssm_stream_t stream);

size_t rssm_gdn_workspace_size(const rssm_gdn_dims* dims);

/* rssm_gdn_precompute -- per-row scalar tables. For row b, value head hv, key head
 * kh, w = row_wp[b], ring entries i < w and the current gate g_t = g[b][hv]:
 *   kk_i = k_i . k_t,  kq_i = k_i . q_t,  kq_t = k_t . q_t   (key head kh)
 *   gamma_i = prod_{j=i+1..w-1} g_j,  Gu = prod_{j<w} g_j,  Go = g_t Gu,
 *   Gamma_i = prod_{j=i+1..w} g_j (with g_w = g_t; Gamma_w = 1)
 * stored per (b, hv) as [gamma_i kk_i (L), Gamma_i kq_i (L), Gamma_i (L), Gu, Go,
 * kq_t, beta_t, g_t, pad]. */
int rssm_gdn_precompute(const rssm_gdn_dims* dims, const void* q, const void* k,
                        const float* beta, const float* g, const void* ring_k,
                        const float* ring_g, const int32_t* cache_indices, const int32_t* row_wp,
                        void* workspace, size_t workspace_bytes, int32_t* dev_err,
                        rssm_stream_t stream);

/* rssm_gdn_output -- fused GDN output / flush ([GDN] 实现拆解 item 1). Streams
 * S0[s][hv] once, computing a = S0 k_t and c = S0 q_t per value row, then
 *   u   = Gu a + sum_{i<w} gamma_i kk_i d_i       (= S_{t-1} k_t)
 *   d_t = beta_t (v_t - g_t u)                     (written to ring_d entry w)
 *   o   = Go c + sum_{i<w} Gamma_i kq_i d_i + kq_t d_t
 * and on flush rows stores S = Go S0 + sum_{i<=w} Gamma_i d_i k_i^T. k_t is read
 * from ring_k entry w (rssm_gdn_ring_append), q_t from q [batch][HK][K]. */
int rssm_gdn_output(const rssm_gdn_dims* dims, float* state, const void* q, const void* v,
                    const void* ring_k, float* ring_d, const int32_t* cache_indices,
                    const int32_t* row_wp, const uint8_t* row_flush, const void* workspace,
                    size_t workspace_bytes, void* o, int32_t* dev_err, rssm_stream_t stream);

/* rssm_gdn_decode -- rssm_gdn_precompute then rssm_gdn_output. */
int rssm_gdn_decode(const rssm_gdn_dims* dims, float* state, const void* q, const void* k,
                    const void* v, const float* beta, const float* g, const void* ring_k,
                    const float* ring_g, float* ring_d, const int32_t* cache_indices,
                    const int32_t* row_wp, const uint8_t* row_flush, void* workspace,
                    size_t workspace_bytes, void* o, int32_t* dev_err, rssm_stream_t stream);

/* rssm_gdn_prepare -- the per-row prologue of one GDN decode step in ONE launch
 * (one CTA per row): the STANDARD cursor step of rssm_advance_cursors (when
 * advance != 0), rssm_gdn_ring_append, then rssm_gdn_precompute; results are
 * those of the three calls in that order ([GDN] 实现拆解 items 1 and 2: the
 * decode kernel's inputs are the ring and per-row cursors with a forced-flush
 * mask). With advance == 0 the row cursors come from an earlier
 * rssm_advance_cursors; slot_wp, force_flush and row_flush are then unused (may
 * be NULL). Arguments, layouts and errors as in those calls. */
int rssm_gdn_prepare(const rssm_gdn_dims* dims, int advance, const uint8_t* force_flush,
                     int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush, const void* q,
                     const void* k, const float* beta, const float* g,
                     const int32_t* cache_indices, void* ring_k, float* ring_g, void* workspace,
                     size_t workspace_bytes, int32_t* dev_err, rssm_stream_t stream);

/* rssm_gdn_step -- one whole GDN ReplaySSM decode step in two launches:
 * rssm_gdn_prepare then rssm_gdn_output. row_flush is always required.
 * Arguments, layouts and errors as in those two calls. */
int rssm_gdn_step(const rssm_gdn_dims* dims, int advance, const uint8_t* force_flush,
                  int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush, float* state,
                  const void* q, const void* k, const void* v, const float* beta, const float* g,
                  const int32_t* cache_indices, void* ring_k, float* ring_g, float* ring_d,
                  void* workspace, size_t workspace_bytes, void* o, int32_t* dev_err,
                  rssm_stream_t stream);

/* rssm_gdn_full_state_decode -- the conventional GDN decode step: read S, apply
 * S <- g S + beta (v - g S k) k^T, write S, o = S q. ring_len is ignored. */
int rssm_gdn_full_state_decode(const rssm_gdn_dims* dims, float* state, const void* q,
                               const void* k, const void* v, const float* beta, const float* g,
                               const int32_t* cache_indices, void* o, int32_t* dev_err,
                               rssm_stream_t stream);

/* ------------------------------------------------------------------------- */
/* KDA: the gated delta rule with a per-key-channel gate                      */
/* ------------------------------------------------------------------------- */

/* [GDN] 实现拆解 item 1: one buffered decode kernel serves the scalar GDN gate and
 * the KDA per-K gate (IS_KDA); 评论区精华: the KDA gate ring is g_cache [slots, HV,
 * L, K] and the report saw no gain for KDA. Reading of the recurrence (the pages
 * print none): the GDN rule with the scalar gate replaced by Diag(a), a in (0, 1]^K
 * per value head:
 *   S <- S Diag(a) + beta (v - S Diag(a) k) k^T,  o = S q.
 * Dims are rssm_gdn_dims (K = 128, V a multiple of 32, L <= 64), fp32 state.
 * Layouts (row-major, dense):
 *   state   [num_slots][HV][V][K] float32  checkpoint S0 per slot
 *   ring_d  [num_slots][HV][V/32][L][32] float32 (as the GDN ring d)
 *   ring_k  [num_slots][HK][L][K] act_dtype
 *   ring_a  [num_slots][HV][L][K] float32  the gates a_i
 *   q, k    [batch][HK][K] act_dtype; v [batch][HV][V] act_dtype
 *   beta    [batch][HV] float32; a [batch][HV][K] float32; o [batch][HV][V] out_dtype
 * Cursors come from rssm_advance_cursors (STANDARD), as for the GDN. */

/* Bytes of workspace rssm_kda_prepare / rssm_kda_output need: per (row, value
 * head) the gated vectors Gam o k_t, Gam o q_t and Gam = prod_{j<=w} a_j, the
 * k_i . (Gam_i o k_t) and k_i . (Gam_i o q_t) tables and beta; then per (row,
 * value head) the gated keys Gam_i o k_i of flush rows. 0 for invalid dims. */
size_t rssm_kda_workspace_size(const rssm_gdn_dims* dims);

/* rssm_kda_prepare -- append a_t into ring_a and k_t into ring_k at entry
 * row_wp[b], and build the tables of the current step (one CTA per (row, value
 * head)). Needs the cursors of the step (row_wp, row_flush). */
int rssm_kda_prepare(const rssm_gdn_dims* dims, const void* q, const void* k, const float* a,
                     const float* beta, const int32_t* cache_indices, const int32_t* row_wp,
                     const uint8_t* row_flush, void* ring_k, float* ring_a, void* workspace,
                     size_t workspace_bytes, int32_t* dev_err, rssm_stream_t stream);

/* rssm_kda_output -- the fused output / flush kernel: streams each (row, value
 * head, 32 value rows) tile of S0 once,
 *   u   = S0 (Gam o k_t) + sum_{i<w} (k_i . (Gam_i o k_t)) d_i,  d_t = beta (v - u),
 *   o   = S0 (Gam o q_t) + sum_{i<=w} (k_i . (Gam_i o q_t)) d_i,
 * (Gam_i = prod_{j=i+1..w} a_j per channel, Gam = prod_{j<=w} a_j), writes d_t into
 * ring_d entry w and, on flush rows, S = S0 Diag(Gam) + sum_{i<=w} d_i (Gam_i o
 * k_i)^T. Needs the tables of rssm_kda_prepare. */
int rssm_kda_output(const rssm_gdn_dims* dims, float* state, const void* v, float* ring_d,
                    const int32_t* cache_indices, const int32_t* row_wp,
                    const uint8_t* row_flush, const void* workspace, size_t workspace_bytes,
                    void* o, int32_t* dev_err, rssm_stream_t stream);

/* rssm_kda_step -- one KDA ReplaySSM decode step: rssm_advance_cursors
 * (STANDARD; skipped when advance == 0), rssm_kda_prepare, rssm_kda_output. */
int rssm_kda_step(const rssm_gdn_dims* dims, int advance, const uint8_t* force_flush,
                  int32_t* slot_wp, int32_t* row_wp, uint8_t* row_flush, float* state,
                  const void* q, const void* k, const void* v, const float* beta, const float* a,
                  const int32_t* cache_indices, void* ring_k, float* ring_a, float* ring_d,
                  void* workspace, size_t workspace_bytes, void* o, int32_t* dev_err,
                  rssm_stream_t stream);

/* rssm_kda_full_state_decode -- the conventional KDA decode step: read S, apply
 * S <- S Diag(a) + beta (v - S Diag(a) k) k^T, write S, o = S q. */
int rssm_kda_full_state_decode(const rssm_gdn_dims* dims, float* state, const void* q,
                               const void* k, const void* v, const float* beta, const float* a,
                               const int32_t* cache_indices, void* o, int32_t* dev_err,
                               rssm_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Gated delta net: speculative verify                                        */
/* ------------------------------------------------------------------------- */

/* Bytes of device workspace rssm_gdn_spec_verify needs for T drafts: per-(row,
 * value head) coefficient tables, then float32 copies of the drafts' keys and
 * queries per (row, key head). 0 for invalid dims or T. */
size_t rssm_gdn_spec_workspace_size(const rssm_gdn_dims* dims, int32_t T);

/* rssm_gdn_spec_verify -- score a linear chain of T draft tokens per row from the
 * checkpoint and the circular ring, without materialising per-draft states
 * ([SPEC] 实现拆解 item 3, gdn_replayssm_spec_circular_kernel), after first
 * folding, for slots whose fold is pending, the committed entries into the
 * checkpoint by replaying the recurrence sequentially from the raw inputs
 * ([SPEC] 实现拆解 item 3, gdn_replayssm_exact_fold_kernel; 评论区精华: the exact
 * fold removed the long-output drift). Two launches: a prologue whose CTAs either
 * fold a pending slot's tile or compute a (row, key head)'s tables (key dot
 * products and gate products, and float32 copies of the drafts' k and q, into
 * `workspace`); then the verify, which also writes the drafts' ring entries.
 *
 * Cursors (read only here; see RSSM_CURSOR_SPEC_COMMIT): slot_wp = cnt,
 * slot_base = base, slot_flush = fold pending. Committed entries sit at ring
 * positions (base + i) % L, i < cnt. With a pending fold the effective history
 * is empty and base' = (base + cnt) % L. Draft j is written at position
 * (base + cnt + j) % L (d, k, g, and the raw v and beta a later fold replays).
 * Draft j's output is that of the recurrence after the history and drafts 0..j;
 * with u_j = S_{m-1} k_j and m = history + j, the chain is evaluated as
 *   u_j = Gu_j (S0 k_j) + sum_{i<m} (prod_{l=i+1..m-1} gate_l)(k_i . k_j) d_i
 *   d_m = beta_j (v_j - g_j u_j)
 *   o_j = Go_j (S0 q_j) + sum_{i<=m} (prod_{l=i+1..m} gate_l)(k_i . q_j) d_i
 * where entries i < history are ring entries and the rest earlier drafts.
 *
 * Inputs per draft: q, k [batch][T][HK][K], v [batch][T][HV][V] (act_dtype),
 * beta, g [batch][T][HV] float32. Output o [batch][T][HV][V] (out_dtype).
 * Extra rings: ring_v [num_slots][HV][L][V] act_dtype (raw v), ring_beta
 * [num_slots][HV][L] float32. ring_k doubles as the raw k ring (the kernel takes k
 * as given; no normalisation happens inside).
 * Errors: RSSM_ERR_CONFIG when T < 1 or L < 2T ([SPEC] 关键源码片段, server_args:
 * the ring must hold at least twice the drafts); RSSM_ERR_UNSUPPORTED for T > 8.
 * A slot whose count breaks cnt + T <= L (without a pending fold) is skipped and
 * flagged RSSM_DEVERR_CURSOR. */
int rssm_gdn_spec_verify(const rssm_gdn_dims* dims, int32_t T, float* state, const void* q,
                         const void* k, const void* v, const float* beta, const float* g,
                         float* ring_d, void* ring_k, float* ring_g, void* ring_v,
                         float* ring_beta, const int32_t* cache_indices, const int32_t* slot_wp,
                         const int32_t* slot_base, const uint8_t* slot_flush, void* workspace,
                         size_t workspace_bytes, void* o, int32_t* dev_err,
                         rssm_stream_t stream);

/* rssm_gdn_spec_full_state_verify -- the conventional speculative verify, built as
 * the in-house comparison for rssm_gdn_spec_verify ([SPEC] 功能与动机: the
 * recurrent verify keeps a full-state snapshot per draft token, the
 * intermediate_ssm buffers). For each row with s >= 0 the T drafts are applied in
 * order to a copy of slot s's state: S_j = g_j S_{j-1} + beta_j (v_j - g_j S_{j-1}
 * k_j) k_j^T, o_j = S_j q_j; S_j is stored as snapshots[b][j] ([batch][T][HV][V][K]
 * float32, caller-allocated, size from rssm_gdn_spec_full_state_snapshot_bytes).
 * The pool is not modified. Inputs, outputs and errors as rssm_gdn_spec_verify
 * (ring_len unused). */
size_t rssm_gdn_spec_full_state_snapshot_bytes(const rssm_gdn_dims* dims, int32_t T);
int rssm_gdn_spec_full_state_verify(const rssm_gdn_dims* dims, int32_t T, const float* state,
                                    const void* q, const void* k, const void* v,
                                    const float* beta, const float* g,
                                    const int32_t* cache_indices, float* snapshots,
                                    size_t snapshot_bytes, void* o, int32_t* dev_err,
                                    rssm_stream_t stream);

/* rssm_gdn_spec_full_state_commit -- the commit of the conventional verify: for each
 * row with s >= 0 and a = num_accepted[b] > 0, state[s] = snapshots[b][a-1]; rows
 * with a = 0 keep their state. a outside 0..T: row skipped, RSSM_DEVERR_CURSOR. */
int rssm_gdn_spec_full_state_commit(const rssm_gdn_dims* dims, int32_t T, float* state,
                                    const float* snapshots, const int32_t* cache_indices,
                                    const int32_t* num_accepted, int32_t* dev_err,
                                    rssm_stream_t stream);

/* ------------------------------------------------------------------------- */

/* rssm_mamba2_materialize_state -- test / debug: the current recurrent state of the
 * dims->batch slots listed in slots[] (negative entries skipped), folded from the
 * checkpoint and the slot's live ring entries 0..c-1 (c = slot_wp[s], the entries
 * written since the last flush) into out [batch][H][P][N] float32, without
 * touching the pool, the rings or the cursors ([M2] 实现拆解 item 1: a flush
 * stores exactly this state):
 *   S = P S0 + sum_{i<c} P_i dt_i x_i B_i^T,  P_i = exp(A_h sum_{i<j<c} dt_j),
 *   P = exp(A_h sum_{j<c} dt_j).
 * Accumulates in fp32 from the stored (possibly bf16) checkpoint; the result is not
 * rounded. Slot or cursor out of range: skipped and flagged in dev_err. Not on the
 * decode path (plain loads, one CTA per (slot, head)). */
int rssm_mamba2_materialize_state(const rssm_mamba2_dims* dims, const void* state,
                                  const float* A, const void* ring_x, const float* ring_dt,
                                  const void* ring_B, const int32_t* slots,
                                  const int32_t* slot_wp, float* out, int32_t* dev_err,
                                  rssm_stream_t stream);

/* rssm_gdn_materialize_state -- test / debug: the GDN counterpart. The live entries
 * of slot s are c = slot_wp[s] entries at ring positions (base + i) % L with base =
 * slot_base[s] (slot_base NULL: base 0, the decode ring; the spec ring passes its
 * cache_base, and a pending fold's entries are included) ([GDN] 实现拆解 item 1;
 * [SPEC] 实现拆解 item 2):
 *   S = G S0 + sum_{i<c} Gamma_i d_i k_i^T,  Gamma_i = prod_{i<j<c} g_j,
 *   G = prod_{j<c} g_j,
 * into out [batch][HV][V][K] float32. Errors as rssm_mamba2_materialize_state. */
int rssm_gdn_materialize_state(const rssm_gdn_dims* dims, const float* state, const void* ring_k,
                               const float* ring_g, const float* ring_d, const int32_t* slots,
                               const int32_t* slot_wp, const int32_t* slot_base, float* out,
                               int32_t* dev_err, rssm_stream_t stream);

/* rssm_debug_umma_fold -- test / debug: the tensor-core building block of the flush
 * folds on its own. D[r][c] = sum_{i<=w} A[r][i] B[i][c] for r < 128, c < N
 * (N = 64 or 128), computed by the 5th-generation tensor cores (tcgen05.mma, the
 * accumulator in tensor memory): A is float32 [128][16] (device, caller owned;
 * entries i > w ignored), split into three bf16 parts whose sum carries its 24-bit
 * significand; B is bf16 [16][N] in the ring layout (entry-major; entries i > w
 * ignored); D float32 [128][N]. 0 <= w < 16. One CTA of 128 threads. The pages have
 * no counterpart: it pins the operand layouts the decode kernels' folds use (the
 * fold itself is the flush of [M2] 实现拆解 item 1 and [GDN] 实现拆解 item 1).
 * Errors: RSSM_ERR_INVALID_ARG (w or N out of range, null or misaligned pointers),
 * RSSM_ERR_CUDA; a completion wait that runs out sets RSSM_DEVERR_TIMEOUT. */
int rssm_debug_umma_fold(const float* A, const uint16_t* B, int w, int N, float* D,
                         int32_t* dev_err, rssm_stream_t stream);

/* rssm_debug_pipeline_copy -- test / debug: exercises the bounded waits of the
 * streaming pipeline every decode kernel runs on. Copies n_tiles tiles of 16 KB
 * from src to dst (float32, device, caller owned, 16-byte aligned) through that
 * pipeline: each tile is staged in shared memory by a 1-D bulk copy whose arrival a
 * stage barrier counts, then written out by the consumer warps. With stall_tile in
 * 0..n_tiles-1 that tile's stage barrier is armed for 16 bytes more than its copy
 * delivers, so it never completes although the copy lands: the waiting warp gives
 * up after wait_us microseconds (1..2000000), ORs RSSM_DEVERR_TIMEOUT into *dev_err
 * (when non-NULL), and its CTA winds down -- the other warps stop waiting, each
 * producer waits (bounded) for the copies it issued -- so the kernel returns with no
 * copy in flight and the context stays usable; dst is then only partly written.
 * stall_tile < 0 copies every tile. The decode kernels wait 2 s before giving up;
 * the pages have no counterpart (failure handling of this library). Errors:
 * RSSM_ERR_INVALID_ARG (n_tiles < 0, stall_tile >= n_tiles, wait_us out of range,
 * null or misaligned src/dst), RSSM_ERR_CUDA. */
int rssm_debug_pipeline_copy(const float* src, float* dst, int n_tiles, int stall_tile,
                             int wait_us, int32_t* dev_err, rssm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RSSM_H */
