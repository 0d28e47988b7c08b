// Per-atom tensor-core step shared by the streaming (few-token) kernels:
// expand one 16-row x 64-k atom of packed codes into mma.sync A fragments and
// multiply it with the matching activation chunk held in shared memory.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

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

// Magnitude-table entry `code` of the table at shared address `lut_s`: the
// address is formed with a multiply-add, which issues on the FMA pipe and
// leaves the integer pipe to the code expansion.
__device__ __forceinline__ Lut lut_entry(uint32_t lut_s, uint32_t code) {
    uint32_t addr;
    asm("mad.lo.u32 %0, %1, 16, %2;" : "=r"(addr) : "r"(code), "r"(lut_s));
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return lut_from_uint4(v);
}

// One shared-memory byte, zero-extended by the load itself (no integer-pipe
// extraction of the two scale codes a lane owns).
__device__ __forceinline__ uint32_t lds_u8(uint32_t saddr) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(saddr));
    return v;
}

// x' = RN(x * s) on a pair of activations: one packed multiply rounds the
// exact product once, as the AWQ pre-quant scale is defined.
template <bool F16>
__device__ __forceinline__ uint32_t awq_mul2(uint32_t x, uint32_t s) {
    uint32_t r;
    if constexpr (F16) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(s));
    else asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(s));
    return r;
}

// Read-only 128-bit global load through L1 (the AWQ scale vector is small and
// shared by every warp of the SM).
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// AWQ on the ring stages of a streaming kernel: x' = RN(x * s) in place on the
// activation rows of a stage (row stride XS elements, rows <= TOK, B 64-k
// blocks of which `xk` k hold data), s = the pre-quant scale at the stage's
// k.  NTHR threads share a stage in 8-element chunks (chunk c: row
// c / kPerRow, column c % kPerRow); each thread loads its chunks' scales one
// stage ahead, so the scale reads never sit between a stage's arrival and its
// MMAs.  The callers synchronise the threads before a stage is read.  Rows
// past M and k past K are left alone (they only meet zero weights or are
// never stored).
template <bool F16, int XS, int TOK, int B, int NTHR>
struct AwqStages {
    static constexpr int kPerRow = B * kBlockK / 8;
    static constexpr int kU = (TOK * kPerRow + NTHR - 1) / NTHR;     // chunks per thread
    uint4 s[kU];

    __device__ __forceinline__ void prefetch(const uint16_t* srow, int rows, int xk, int t) {
        #pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int c = t + u * NTHR, col = c % kPerRow;
            if (c < rows * kPerRow && col * 8 < xk) s[u] = ldg_nc_v4(srow + col * 8);
        }
    }

    __device__ __forceinline__ void apply(uint16_t* xs, int rows, int xk, int t) const {
        #pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int c = t + u * NTHR, r = c / kPerRow, col = c % kPerRow;
            if (c < rows * kPerRow && col * 8 < xk) {
                uint4* px = reinterpret_cast<uint4*>(xs + r * XS + col * 8);
                uint4 xv = *px;
                xv = make_uint4(awq_mul2<F16>(xv.x, s[u].x), awq_mul2<F16>(xv.y, s[u].y),
                                awq_mul2<F16>(xv.z, s[u].z), awq_mul2<F16>(xv.w, s[u].w));
                *px = xv;
            }
        }
    }
};

// One atom: a lane holds 16 code bytes (rows g and g+8 of the atom, group q)
// and their two scale codes sc0 (row g) and sc1 (row g+8); xrow points at
// token row g, group q of the activation chunk (row stride XS elements,
// 16-byte aligned).  Within the group the MMA's k order is permuted -- MMA j
// consumes k = 4j..4j+3 of every lane's group -- and the activation fragments
// use the same permutation.  Only the first `mt_used` 8-token tiles hold
// tokens (warp-uniform): the MMAs and activation loads of the others are
// skipped, their accumulators stay zero.
template <int MT, int XS, bool F16>
__device__ __forceinline__ void atom_mma(const uint4 codes, uint32_t sc0, uint32_t sc1, uint32_t lut_s,
                                         const uint16_t* xrow, float acc[MT][4], int mt_used = MT) {
    const Lut t0 = lut_entry(lut_s, sc0);
    const Lut t1 = lut_entry(lut_s, sc1);
    uint32_t ra[8], rb[8];
    expand8(codes.x, t0, ra);
    expand8(codes.y, t0, ra + 4);
    expand8(codes.z, t1, rb);
    expand8(codes.w, t1, rb + 4);
    #pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        if (mt >= mt_used) break;
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

// One ring stage of B 64-k blocks (block stride BLK bytes; this warp's atom at
// `a`, its activation chunk at `xrow`), nb of them holding data, the first
// `mt_used` 8-token tiles holding tokens.  Full stages take a loop without
// per-block bounds checks; only the last stage of a K slice can be partial.
template <int MT, int XS, bool F16, int B, uint32_t BLK>
__device__ __forceinline__ void stage_mma(const uint8_t* a, int lane, uint32_t lut_s, const uint16_t* xrow,
                                          int nb, float acc[MT][4], int mt_used = MT) {
    uint4 codes[B];
    uint32_t s0[B], s1[B];
    const uint32_t sa = smem_u32(a) + kAtomCodeBytes + 2 * lane;
    #pragma unroll
    for (int b = 0; b < B; ++b) {
        codes[b] = *reinterpret_cast<const uint4*>(a + b * BLK + 16 * lane);
        s0[b] = lds_u8(sa + b * BLK);
        s1[b] = lds_u8(sa + b * BLK + 1);
    }
    if (nb >= B) {
        #pragma unroll
        for (int b = 0; b < B; ++b)
            atom_mma<MT, XS, F16>(codes[b], s0[b], s1[b], lut_s, xrow + b * kBlockK, acc, mt_used);
    } else {
        #pragma unroll
        for (int b = 0; b < B; ++b)
            if (b < nb) atom_mma<MT, XS, F16>(codes[b], s0[b], s1[b], lut_s, xrow + b * kBlockK, acc, mt_used);
    }
}

}  // namespace nvfp4
