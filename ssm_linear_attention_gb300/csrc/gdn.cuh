// gdn.cuh -- what the gated-delta-net decode translation units share: tile shape,
// coefficient-table row length and the dims check.
#pragma once

#include "rssm.h"

namespace rssm {
namespace gdn {

constexpr int KD = 128;  // key dim handled by these kernels
constexpr int VB = 32;   // value rows per work item (a 16 KB fp32 tile)
constexpr int TILE = VB * KD * 4;

// Per-(row, value head) table: gamma_i (k_i.k_t), Gamma_i (k_i.q_t), Gamma_i
// (i < L), Gu, Go, k_t.q_t, beta_t, g_t, padded to 4 floats.
__host__ __device__ inline int tbl_floats(int L) { return (3 * L + 5 + 3) & ~3; }

// Host-side validation of a dims struct (RSSM_OK or an error status).
int check_dims(const rssm_gdn_dims* d);

}  // namespace gdn
}  // namespace rssm
