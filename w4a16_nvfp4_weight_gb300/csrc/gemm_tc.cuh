// Launch interface of the tensor-core (tcgen05) tile GEMM for larger M.
#pragma once
#include "common.cuh"

namespace nvfp4 {

struct TcParams {
    const uint16_t* X;        // BF16 [M, K]
    const uint16_t* pqs;      // BF16 [K] or nullptr
    const uint8_t* rp;        // repacked weight
    uint16_t* Y;              // BF16 [M, N]
    int64_t M, N, K;
    void* workspace;
    size_t workspace_bytes;
    int* status;
};

// Shape rule between the decode kernel and the tile kernel.
bool use_tc_path(int64_t M);
size_t tc_workspace_bytes(int64_t M, int64_t N, int64_t K, bool has_pqs);
nvfp4_status launch_tc(const TcParams& p, cudaStream_t stream);

}  // namespace nvfp4
