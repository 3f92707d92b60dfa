// slots.cu -- slot fork: copy whole per-slot records (checkpoint, rings, cursors)
// from source slots to destination slots.
//
// "GDN ReplaySSM decode (Part A of RFC 28511)", 实现拆解 item 3 and 评论区精华: the
// memory pool's copy_from copies the ring buffers along with the state and sets
// the cursors, and the review notes that copying a slot whose ring still holds
// live entries must carry them too. Here every per-slot buffer the caller lists is
// copied whole, cursors included, so the destination continues exactly as the
// source would: the fork needs no flushed source.
#include "common.cuh"
#include "internal.h"

namespace rssm {
namespace slots {

constexpr int kThreads = 256;
constexpr int kChunk = 16384;  // bytes one CTA copies per work item

struct Args {
    char* base[RSSM_MAX_SLOT_BUFFERS];
    unsigned long long slot_bytes[RSSM_MAX_SLOT_BUFFERS];
    int first_chunk[RSSM_MAX_SLOT_BUFFERS + 1];  // prefix sums of chunks per slot record
    int vec16[RSSM_MAX_SLOT_BUFFERS];            // 16-byte copies (base and size aligned)
    int nbuf;
    const int32_t* src;
    const int32_t* dst;
    int n, num_slots;
    int32_t* dev_err;
};

__global__ void __launch_bounds__(kThreads) copy_slots_kernel(const Args a) {
    const int per = a.first_chunk[a.nbuf];
    const long items = (long)a.n * per;
    for (long it = blockIdx.x; it < items; it += gridDim.x) {
        const int pair = (int)(it / per);
        const int r = (int)(it - (long)pair * per);
        const int s = a.src[pair], d = a.dst[pair];
        if (s < 0 || d < 0) continue;  // padding
        if (s >= a.num_slots || d >= a.num_slots) {
            if (threadIdx.x == 0 && r == 0) set_dev_err(a.dev_err, RSSM_DEVERR_SLOT);
            continue;
        }
        if (s == d) continue;
        int b = 0;
        while (r >= a.first_chunk[b + 1]) ++b;
        const unsigned long long sb = a.slot_bytes[b];
        const unsigned long long off = (unsigned long long)(r - a.first_chunk[b]) * kChunk;
        const unsigned long long len = sb - off < (unsigned long long)kChunk ? sb - off : kChunk;
        const char* from = a.base[b] + (unsigned long long)s * sb + off;
        char* to = a.base[b] + (unsigned long long)d * sb + off;
        if (a.vec16[b]) {
            const uint4* f4 = reinterpret_cast<const uint4*>(from);
            uint4* t4 = reinterpret_cast<uint4*>(to);
            const int nv = (int)(len >> 4);
            constexpr int U = kChunk / 16 / kThreads;  // 16-byte words per thread
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = threadIdx.x + u * kThreads;
                if (i < nv) v[u] = f4[i];
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = threadIdx.x + u * kThreads;
                if (i < nv) t4[i] = v[u];
            }
        } else {
            for (int i = threadIdx.x; i < (int)len; i += kThreads) to[i] = from[i];
        }
    }
}

}  // namespace slots
}  // namespace rssm

using namespace rssm;

extern "C" int rssm_copy_slots(const rssm_slot_buffer* buffers, int32_t n_buffers,
                               const int32_t* src_slots, const int32_t* dst_slots, int32_t n,
                               int32_t num_slots, int32_t* dev_err, rssm_stream_t stream) {
    if (!buffers || n_buffers < 1 || n_buffers > RSSM_MAX_SLOT_BUFFERS || n < 0 || num_slots <= 0)
        return RSSM_ERR_INVALID_ARG;
    slots::Args a{};
    int chunks = 0;
    for (int b = 0; b < n_buffers; ++b) {
        const rssm_slot_buffer& sb = buffers[b];
        if (sb.base == nullptr || sb.slot_bytes == 0) return RSSM_ERR_INVALID_ARG;
        const unsigned long long c = (sb.slot_bytes + slots::kChunk - 1) / slots::kChunk;
        if (c > (1u << 20)) return RSSM_ERR_INVALID_ARG;  // > 16 GB per slot record
        a.base[b] = static_cast<char*>(sb.base);
        a.slot_bytes[b] = sb.slot_bytes;
        a.vec16[b] = aligned16(sb.base) && (sb.slot_bytes & 15) == 0;
        a.first_chunk[b] = chunks;
        chunks += (int)c;
        if (chunks > (1 << 24)) return RSSM_ERR_INVALID_ARG;
    }
    a.first_chunk[n_buffers] = chunks;
    if (n == 0) return RSSM_OK;
    if (!ok_ptr(src_slots) || !ok_ptr(dst_slots)) return RSSM_ERR_INVALID_ARG;
    a.nbuf = n_buffers;
    a.src = src_slots;
    a.dst = dst_slots;
    a.n = n;
    a.num_slots = num_slots;
    a.dev_err = dev_err;
    DeviceInfo di;
    if (!device_info(&di)) return RSSM_ERR_CUDA;
    const long items = (long)n * chunks;
    long grid = (long)di.sm_count * 8;
    if (grid > items) grid = items;
    slots::copy_slots_kernel<<<(unsigned)grid, slots::kThreads, 0, (cudaStream_t)stream>>>(a);
    return launch_status();
}
