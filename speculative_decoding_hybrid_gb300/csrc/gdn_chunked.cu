// Chunked GatedDeltaNet prefill -- placeholder until the kernel lands.
#include "common.cuh"

extern "C" size_t gdn_prefill_workspace_bytes(const gdn_dims *, int32_t, int32_t) { return 0; }

extern "C" int gdn_chunked_prefill(const gdn_dims *, int32_t, int32_t, const int32_t *, int32_t, const gdn_bf16 *,
                                   const gdn_bf16 *, const gdn_bf16 *, const float *, const float *, float *,
                                   int64_t, int32_t, const int32_t *, const int32_t *, gdn_bf16 *, int32_t, void *,
                                   size_t, uint32_t *, void *) {
    return GDN_ERR_ARG;
}
