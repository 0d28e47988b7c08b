// Tensor-core tile GEMM (placeholder until the tcgen05 kernel lands).
#include "common.cuh"
#include "gemm_tc.cuh"

namespace nvfp4 {

bool use_tc_path(int64_t) { return false; }
size_t tc_workspace_bytes(int64_t, int64_t, int64_t, bool) { return 0; }
nvfp4_status launch_tc(const TcParams&, cudaStream_t) {
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "tile GEMM not available");
}

}  // namespace nvfp4
