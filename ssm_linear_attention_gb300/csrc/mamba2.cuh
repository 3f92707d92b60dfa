// mamba2.cuh -- what the Mamba2 translation units share: the coefficient-table
// row length and the dims check.
#pragma once

#include <cuda_runtime.h>

#include "rssm.h"

namespace rssm {
namespace m2 {

// Per-(row, head) table: coef_0..coef_{L-1}, a_0..a_{L-1}, Pm1, padded to 4 floats.
__host__ __device__ inline int tbl_floats(int L) { return (2 * L + 1 + 3) & ~3; }

// Workspace: the tables [batch][H][tbl_floats(L)] float32, then (at a 256-byte
// boundary) the output kernel's work counter, two unsigned words that the prologue
// kernels zero every step and the output kernel leaves at zero.
__host__ __device__ inline size_t sched_offset(int batch, int H, int L) {
    return ((size_t)batch * H * tbl_floats(L) * 4 + 255) & ~(size_t)255;
}
constexpr size_t kSchedBytes = 256;
// Words kRowCountWord.. of that block: the one-launch small-batch step's per-row
// counters (zero before the workspace's first use; the step leaves them zero).
constexpr int kRowCountWord = 16;
constexpr int kSmallStepMaxBatch = 16;   // batches the one-launch step takes
constexpr int kSmallStepMaxRing = 64;

// Host-side validation of a dims struct (RSSM_OK or an error status).
int check_dims(const rssm_mamba2_dims* d);

}  // namespace m2

// The one-launch Mamba2 step for small batches (mamba2_small.cu); RSSM_ERR_UNSUPPORTED
// when the shape has no instance.
int m2_step_small(const rssm_mamba2_dims* d, const uint8_t* force_flush, int32_t* slot_wp,
                  int32_t* row_wp, uint8_t* row_flush, void* state, const void* x,
                  const float* dt_raw, const float* dt_bias, int dt_softplus, const float* A,
                  const void* B, const void* C, const float* D, const void* z,
                  const int32_t* cache_indices, void* ring_x, float* ring_dt, void* ring_B,
                  void* workspace, void* y, int32_t* dev_err, cudaStream_t stream);
}  // namespace rssm
