// cursor.cuh -- the STANDARD cursor step of one decode row, shared by the cursor
// kernel and the fused per-row prologue kernels.
//
// [M2] "ReplaySSM: cache SSM inputs for faster Mamba2 standard decode", 实现拆解
// item 3 (per-row write_pos and is_flush); [GDN] "GDN ReplaySSM decode (Part A of
// RFC 28511)", 实现拆解 item 2 (a forced flush per row).
#pragma once

#include "common.cuh"

namespace rssm {

// Row b with slot s = cache_indices[b]: w = slot_wp[s], f = (w == L-1) || force[b];
// row_wp[b] = w, row_flush[b] = f, slot_wp[s] = f ? 0 : w + 1. Padding rows
// (s < 0) and invalid rows (slot or cursor out of range, reported in dev_err) get
// row_wp = 0, row_flush = 0 and return -1; otherwise returns w.
__device__ __forceinline__ int standard_cursor(int b, int s, int num_slots, int L,
                                               int32_t* slot_wp, const uint8_t* force,
                                               int32_t* row_wp, uint8_t* row_flush,
                                               int32_t* dev_err) {
    if (s < 0 || s >= num_slots) {
        if (s >= num_slots) set_dev_err(dev_err, RSSM_DEVERR_SLOT);
        row_wp[b] = 0;
        row_flush[b] = 0;
        return -1;
    }
    const int w = slot_wp[s];
    if (w < 0 || w >= L) {
        set_dev_err(dev_err, RSSM_DEVERR_CURSOR);
        row_wp[b] = 0;
        row_flush[b] = 0;
        return -1;
    }
    const int f = (w == L - 1) || (force != nullptr && force[b] != 0);
    row_wp[b] = w;
    row_flush[b] = static_cast<uint8_t>(f);
    slot_wp[s] = f ? 0 : w + 1;
    return w;
}

// The row's write position from an earlier cursor advance (layers sharing one
// advance): -1 for padding and invalid rows (reported in dev_err).
__device__ __forceinline__ int given_cursor(int b, int s, int num_slots, int L,
                                            const int32_t* row_wp, int32_t* dev_err) {
    if (s < 0) return -1;
    if (s >= num_slots) {
        set_dev_err(dev_err, RSSM_DEVERR_SLOT);
        return -1;
    }
    const int w = row_wp[b];
    if (w < 0 || w >= L) {
        set_dev_err(dev_err, RSSM_DEVERR_CURSOR);
        return -1;
    }
    return w;
}

}  // namespace rssm
