// mamba2.cuh -- what the Mamba2 translation units share: the coefficient-table
// row length and the dims check.
#pragma once

#include "rssm.h"

namespace rssm {
namespace m2 {

// Per-(row, head) table: coef_0..coef_{L-1}, a_0..a_{L-1}, Pm1, padded to 4 floats.
__host__ __device__ inline int tbl_floats(int L) { return (2 * L + 1 + 3) & ~3; }

// Host-side validation of a dims struct (RSSM_OK or an error status).
int check_dims(const rssm_mamba2_dims* d);

}  // namespace m2
}  // namespace rssm
