// gdn_pending.cu -- gated-delta-net entry points not yet implemented in this build:
// they validate nothing and return RSSM_ERR_UNSUPPORTED.
#include "rssm.h"

extern "C" int rssm_gdn_ring_append(const rssm_gdn_dims*, const void*, const float*, const int32_t*,
                                    const int32_t*, void*, float*, int32_t*, rssm_stream_t) {
    return RSSM_ERR_UNSUPPORTED;
}
extern "C" size_t rssm_gdn_workspace_size(const rssm_gdn_dims*) { return 0; }
extern "C" int rssm_gdn_precompute(const rssm_gdn_dims*, const void*, const void*, const float*,
                                   const float*, const void*, const float*, const int32_t*,
                                   const int32_t*, void*, size_t, int32_t*, rssm_stream_t) {
    return RSSM_ERR_UNSUPPORTED;
}
extern "C" int rssm_gdn_output(const rssm_gdn_dims*, float*, const void*, const void*, float*,
                               const int32_t*, const int32_t*, const uint8_t*, const void*, size_t,
                               void*, int32_t*, rssm_stream_t) {
    return RSSM_ERR_UNSUPPORTED;
}
extern "C" int rssm_gdn_decode(const rssm_gdn_dims*, float*, const void*, const void*, const void*,
                               const float*, const float*, const void*, const float*, float*,
                               const int32_t*, const int32_t*, const uint8_t*, void*, size_t, void*,
                               int32_t*, rssm_stream_t) {
    return RSSM_ERR_UNSUPPORTED;
}
extern "C" int rssm_gdn_full_state_decode(const rssm_gdn_dims*, float*, const void*, const void*,
                                          const void*, const float*, const float*, const int32_t*,
                                          void*, int32_t*, rssm_stream_t) {
    return RSSM_ERR_UNSUPPORTED;
}
extern "C" int rssm_gdn_spec_verify(const rssm_gdn_dims*, int32_t, float*, const void*, const void*,
                                    const void*, const float*, const float*, float*, void*, float*,
                                    void*, float*, const int32_t*, const int32_t*, const int32_t*,
                                    const uint8_t*, void*, int32_t*, rssm_stream_t) {
    return RSSM_ERR_UNSUPPORTED;
}
