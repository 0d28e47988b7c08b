// Launch interface of the tensor-core (tcgen05) tile GEMM for larger M.
#pragma once
#include "common.cuh"

namespace nvfp4 {

struct TcParams {
    const uint16_t* X;        // BF16 or FP16 [M, K]
    const uint16_t* pqs;      // [K] or nullptr, same type as X
    const uint8_t* rp;        // repacked weight
    uint16_t* Y;              // [M, N], same type as X
    bool f16;                 // FP16 activations and output (else BF16)
    int64_t M, N, K;
    void* workspace;
    size_t workspace_bytes;
    int* status;
};

// Grouped MoE use of the tile kernel: work items of up to 128*subm permuted
// rows of one expert; X rows are already in permuted (expert-contiguous) order.
struct TcMoeParams {
    bool fc1;                 // FC1 (-> H) or FC2 (x p -> Yp)
    int act;                  // FC1: 0 = gated (gate/up + SwiGLU), 1 = relu2, 2 = silu (non-gated)
    size_t half_stride;       // gated FC1: 0, or bytes from the gate shard to the up shard
    bool f16;                 // FP16 activations (else BF16)
    int subm;                 // 1 or 2: 128 or 256 rows per work item
    const uint16_t* X;        // [x_rows, K] BF16 or FP16, permuted rows
    int64_t x_rows;
    const uint8_t* w;         // stacked repacked experts
    size_t w_stride;
    int64_t N, K, I;          // weight rows (gated FC1: 2I, or I per shard), inner dimension, intermediate size
    const int4* items;        // null: one dense weight, items are runs of 128*subm rows
    const int32_t* n_items;
    int64_t max_items;
    int64_t rows;             // dense use: token rows
    const int32_t* perm;
    const float* wts;
    uint16_t* H;              // FC1 output [x_rows, I]
    float* Yp;                // FC2 output [slots, N]
    int* status;
};
nvfp4_status launch_tc_moe(const TcMoeParams& p, cudaStream_t stream);

// Shape rule between the streaming (decode) kernel and the tile kernels for
// M > 16: the one a cost model predicts faster (always tiles from M = 512).
bool use_tc_path(int64_t M, int64_t N, int64_t K);
// Whether the tile grid alone (no K split) fills at least half of the SMs, or
// M >= 512: the rule of the callers whose tile modes do not split K.
bool tc_tiles_fill(int64_t M, int64_t N);
// The dense tile plan of an M x N x K GEMM: the tensor-memory-A kernel (wa) or
// the shared-memory-operand one, its tokens per tile and its K splits.
void tc_plan_info(int64_t M, int64_t N, int64_t K, bool* wa, int* tokens, int* splits);
size_t tc_workspace_bytes(int64_t M, int64_t N, int64_t K, bool has_pqs);
nvfp4_status launch_tc(const TcParams& p, cudaStream_t stream);

}  // namespace nvfp4
