// Grouped top-k MoE layer (placeholder until the routed-expert kernels land).
#include "common.cuh"

using namespace nvfp4;

extern "C" size_t nvfp4_w4a16_moe_workspace(int64_t, int, int, int64_t, int64_t) { return 0; }

extern "C" nvfp4_status nvfp4_w4a16_moe_grouped(const void*, const float*, const void*, const void*,
                                                const void*, int64_t, int, int, int64_t, int64_t,
                                                void*, int32_t*, float*, int32_t*, int32_t*,
                                                void*, size_t, void*) {
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "nvfp4_w4a16_moe_grouped: not available");
}
