// mamba2.cuh -- what the Mamba2 translation units share: the coefficient-table
// row length and the dims check.
#pragma once

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

// Host-side validation of a dims struct (RSSM_OK or an error status).
int check_dims(const rssm_mamba2_dims* d);

}  // namespace m2
}  // namespace rssm
