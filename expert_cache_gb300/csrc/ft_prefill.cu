// Prefill of one layer: full-layer double buffering and the FP4 grouped GEMMs.
#include <cstdio>
#include "ft_internal.cuh"

extern "C" ft_status ft_moe_prefill_layer(ft_cache* c, int32_t layer, const void* x,
                                          const int32_t* topk_ids, const float* topk_w,
                                          int32_t T, int32_t k, float* y, int32_t flags,
                                          void* debug_h, void* stream) {
    (void)layer; (void)x; (void)topk_ids; (void)topk_w; (void)T; (void)k; (void)y;
    (void)flags; (void)debug_h; (void)stream;
    if (c) snprintf(c->err, sizeof(c->err), "prefill is not available in this build");
    return FT_ERR_STATE;
}
