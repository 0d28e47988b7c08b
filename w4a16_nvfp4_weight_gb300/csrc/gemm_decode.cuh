// Launch interface of the split-K decode GEMM (few tokens).
#pragma once
#include "common.cuh"

namespace nvfp4 {

struct DecodeParams {
    const uint16_t* X;        // BF16 or FP16 [M, K]
    const uint16_t* pqs;      // AWQ pre-quant scale [K] in the activation type, or null
    const uint8_t* rp;        // repacked weight
    uint16_t* Y;              // BF16 or FP16 [M, N]
    int64_t M, N, K;
    int64_t KB;               // 64-k blocks of the padded K
    int kbs;                  // 64-k blocks per split
    int splits;               // CTAs per cluster along K (<= 16)
    int* status;              // device status word
};

// Shared-memory ring shapes: the deep ring streams long K slices; the
// shallow one lets more CTAs share an SM when each CTA's slice is short, so
// that one CTA's pipeline fill and reduction overlap another's work.
enum DecodeRing { kRingDeep = 0, kRingShallow = 1 };

// Dynamic shared memory of one CTA for MT token tiles of 8, the given ring and
// W consumer warps (8: 128 weight rows per CTA; 4: 64 rows).
size_t decode_smem_bytes(int MT, int ring, int W);

// CTAs of the decode kernel that fit on one SM at once (shared memory,
// thread and register bound) for the given activation type and AWQ choice.
int decode_ctas_per_sm(int MT, int ring, int W, bool f16, bool awq);

// Registers per thread of that decode kernel instance (0 if unknown).
int decode_kernel_regs(int MT, int ring, int W, bool f16, bool awq);

// MT = 1 (up to 8 tokens per CTA) or 2 (up to 16); tokens beyond 8*MT are
// covered by a third grid dimension.  W = 8 or 4 consumer warps.
// f16: FP16 activations and output (else BF16).
nvfp4_status launch_decode(const DecodeParams& p, int MT, int ring, int W, bool f16, cudaStream_t stream);

// Xs = RN(X * pqs) in the activation type (FP16 when f16, else BF16) for an
// M x K activation (K a multiple of 16).
nvfp4_status launch_awq_scale(const uint16_t* X, const uint16_t* pqs, uint16_t* Xs, int64_t M, int64_t K,
                              bool f16, cudaStream_t stream);

}  // namespace nvfp4
