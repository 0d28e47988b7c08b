// Per-atom tensor-core step shared by the streaming (few-token) kernels:
// expand one 16-row x 64-k atom of packed codes into mma.sync A fragments and
// multiply it with the matching activation chunk held in shared memory.
#pragma once

#include "common.cuh"

namespace nvfp4 {

// Shared-memory ring of the streaming kernels: kStages stages, each holding
// kBlocksPerStage 64-k blocks of 16*W weight rows (W x 576 contiguous bytes
// each; W consumer warps of 16 rows) followed by the activation chunk of 8*MT
// token rows (row stride padded by 16 bytes so that the rows fall on different
// banks).
constexpr uint32_t kStreamBlockBytes = 8 * kAtomBytes;   // the 128-row block

template <int MT, int S, int B, int W = 8> struct StreamRing {
    static constexpr int kTok = 8 * MT;
    static constexpr int kStages = S;
    static constexpr int kBlocksPerStage = B;
    static constexpr uint32_t kBlockBytes = W * kAtomBytes;
    static constexpr uint32_t kWeightStageBytes = B * kBlockBytes;
    static constexpr int kXRowElems = B * kBlockK + 8;
    static constexpr size_t kXStageBytes = (size_t)kTok * kXRowElems * 2;
    static constexpr size_t kStageBytes = kWeightStageBytes + kXStageBytes;
    static_assert(kStageBytes % 16 == 0 && (kXRowElems * 2) % 16 == 0, "bulk copies need 16-byte alignment");
};

// D += A * B on 16-bit operands of the activation type (BF16, or FP16 when
// F16), FP32 accumulators.
template <bool F16>
__device__ __forceinline__ void mma_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    if constexpr (F16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// One atom: a lane holds 16 code bytes (rows g and g+8 of the atom, group q)
// and the two scale codes; xrow points at token row g, group q of the
// activation chunk (row stride XS elements, 16-byte aligned).  Within the
// group the MMA's k order is permuted -- MMA j consumes k = 4j..4j+3 of every
// lane's group -- and the activation fragments use the same permutation.
template <int MT, int XS, bool F16>
__device__ __forceinline__ void atom_mma(const uint4 codes, uint32_t sc2, const uint4* lut,
                                         const uint16_t* xrow, float acc[MT][4]) {
    const Lut t0 = lut_from_uint4(lut[sc2 & 0xFF]);
    const Lut t1 = lut_from_uint4(lut[(sc2 >> 8) & 0xFF]);
    uint32_t ra[8], rb[8];
    expand8(codes.x, t0, ra);
    expand8(codes.y, t0, ra + 4);
    expand8(codes.z, t1, rb);
    expand8(codes.w, t1, rb + 4);
    #pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const uint4 b01 = *reinterpret_cast<const uint4*>(xrow + mt * 8 * XS);
        const uint4 b23 = *reinterpret_cast<const uint4*>(xrow + mt * 8 * XS + 8);
        const uint32_t a0[4] = {ra[0], rb[0], ra[1], rb[1]};
        const uint32_t a1[4] = {ra[2], rb[2], ra[3], rb[3]};
        const uint32_t a2[4] = {ra[4], rb[4], ra[5], rb[5]};
        const uint32_t a3[4] = {ra[6], rb[6], ra[7], rb[7]};
        mma_16816<F16>(acc[mt], a0, b01.x, b01.y);
        mma_16816<F16>(acc[mt], a1, b01.z, b01.w);
        mma_16816<F16>(acc[mt], a2, b23.x, b23.y);
        mma_16816<F16>(acc[mt], a3, b23.z, b23.w);
    }
}

}  // namespace nvfp4
