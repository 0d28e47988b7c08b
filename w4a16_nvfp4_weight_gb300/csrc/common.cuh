// Shared device/host definitions of the W4A16 NVFP4 library (sm_103a).
//
// The repacked weight layout (documented in include/nvfp4_w4a16.h) and the
// register-level expansion of packed E2M1 codes into BF16 operands live here,
// so that the standalone dequant and every GEMM kernel feed the tensor cores
// exactly the same bits.
#pragma once

#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>

#include "nvfp4_w4a16.h"

namespace nvfp4 {

// ---------------------------------------------------------------- layout ---
constexpr uint32_t kMagic = 0x34504E56u;   // "VNP4"
constexpr uint32_t kVersion = 2;            // 2: BF16 and FP16 magnitude tables
constexpr int kGroup = 16;                  // K elements per E4M3 scale
constexpr int kTileRows = 256;              // rows per tile (N padding)
constexpr int kBlockK = 64;                 // k per atom (K padding)
constexpr int kAtomRows = 16;               // rows per atom
constexpr int kAtomsPerTileK = kTileRows / kAtomRows;   // 16
constexpr int kAtomCodeBytes = 512;         // 16 rows x 64 k x 4 bits
constexpr int kAtomScaleBytes = 64;         // 16 rows x 4 groups
constexpr int kAtomBytes = kAtomCodeBytes + kAtomScaleBytes;   // 576
constexpr size_t kHeaderBytes = 256;
constexpr size_t kLutBytes = 256 * 16;                          // one magnitude table
constexpr size_t kLutBf16Offset = kHeaderBytes;                 // table for BF16 activations
constexpr size_t kLutF16Offset = kHeaderBytes + kLutBytes;      // table for FP16 activations
constexpr size_t kTilesOffset = kHeaderBytes + 2 * kLutBytes;   // 8448

// Byte offset of the magnitude table for the activation type (FP16 or BF16).
template <bool F16>
__host__ __device__ constexpr size_t lut_offset() { return F16 ? kLutF16Offset : kLutBf16Offset; }

struct Header {
    uint32_t magic;
    uint32_t version;
    int64_t N, K, Np, Kp;
    float g;
    float global_scale;
    uint32_t global_is_divisor;
    uint32_t pad_;
};
static_assert(sizeof(Header) <= kHeaderBytes, "header too large");

__host__ __device__ inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Byte offset of atom (tile nt, k-block kb, row-block rb) from the tiles start.
__host__ __device__ inline size_t atom_offset(int64_t nt, int64_t kb, int64_t rb, int64_t KB) {
    return (size_t)(((nt * KB + kb) * kAtomsPerTileK + rb) * kAtomBytes);
}

// ----------------------------------------------------- register expansion ---
// One magnitude-table entry: the 8 E2M1 magnitudes times one E4M3 scale times
// g, rounded to the 16-bit activation type (BF16 or FP16; both keep the sign
// in bit 15), split into low bytes (l0: m0..m3, l1: m4..m7) and high bytes
// (h0, h1), so that one byte permute per byte plane looks up 4 codes.
struct Lut {
    uint32_t l0, l1, h0, h1;
};

__device__ __forceinline__ Lut lut_from_uint4(uint4 v) { return Lut{v.x, v.y, v.z, v.w}; }

// Expand one 32-bit code word (8 consecutive k, sign-split nibble format) to
// four BF16x2 registers: r[0] = (e0, e1), r[1] = (e2, e3), r[2] = (e4, e5),
// r[3] = (e6, e7).  The magnitude of e_i sits in bits 4i..4i+2 (a byte-permute
// selector once bit 3 of every nibble is masked off); the signs of e0..e3 sit
// in bits 7, 15, 23, 31 and those of e4..e7 in bits 3, 11, 19, 27, i.e. on (or
// 4 below) the top bit of each byte of the high-byte planes, where one XOR
// applies them.  XOR (not OR) so that a negative scale or global flips the sign
// as the exact product would.  About 14 integer instructions per 8 weights.
__device__ __forceinline__ void expand8(uint32_t w, const Lut& t, uint32_t r[4]) {
    // The sign shift is written as a multiply so that it can issue on the FMA
    // pipe; the byte permutes and logic ops all need the integer pipe.  Of the
    // forms tried for the two selectors (one shared mask, a multiply-high for
    // the shift) this plain one timed fastest on GB300.
    const uint32_t selA = w & 0x7777u;
    const uint32_t selB = (w >> 16) & 0x7777u;
    const uint32_t loA = __byte_perm(t.l0, t.l1, selA);
    const uint32_t hiA = __byte_perm(t.h0, t.h1, selA) ^ (w & 0x80808080u);
    const uint32_t loB = __byte_perm(t.l0, t.l1, selB);
    const uint32_t hiB = __byte_perm(t.h0, t.h1, selB) ^ ((w * 16u) & 0x80808080u);   // (w << 4)
    r[0] = __byte_perm(loA, hiA, 0x5140);
    r[1] = __byte_perm(loA, hiA, 0x7362);
    r[2] = __byte_perm(loB, hiB, 0x5140);
    r[3] = __byte_perm(loB, hiB, 0x7362);
}

// Streaming 128-bit load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// 16-bit streaming load into a 32-bit register (zero-extended by the load
// itself, so no conversion instruction waits on it right after issue).
__device__ __forceinline__ uint32_t ldg_u16(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// BF16 (bits) of x * s, both BF16: the product is exact in FP32 for normal
// operands, so one RN conversion gives the single-rounded AWQ activation.
__device__ __forceinline__ uint16_t awq_mul_bf16(uint16_t x, uint16_t s) {
    const float xf = __uint_as_float((uint32_t)x << 16);
    const float sf = __uint_as_float((uint32_t)s << 16);
    const float p = __fmul_rn(xf, sf);
    uint16_t out;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(out) : "f"(p));
    return out;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    uint16_t out;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(out) : "f"(v));
    return out;
}

__device__ __forceinline__ uint16_t f32_to_f16_bits(float v) {
    uint16_t out;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(out) : "f"(v));
    return out;
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
    float out;
    asm("cvt.f32.f16 %0, %1;" : "=f"(out) : "h"(h));
    return out;
}

// FP16 (bits) of x * s, both FP16: 11 x 11 significant bits are exact in FP32
// (FP16 subnormals are FP32 normals), so one RN conversion rounds once.
__device__ __forceinline__ uint16_t awq_mul_f16(uint16_t x, uint16_t s) {
    return f32_to_f16_bits(__fmul_rn(f16_bits_to_f32(x), f16_bits_to_f32(s)));
}

// Round an FP32 result to the activation type.
template <bool F16>
__device__ __forceinline__ uint16_t f32_to_act_bits(float v) {
    return F16 ? f32_to_f16_bits(v) : f32_to_bf16_bits(v);
}

template <bool F16>
__device__ __forceinline__ uint16_t awq_mul(uint16_t x, uint16_t s) {
    return F16 ? awq_mul_f16(x, s) : awq_mul_bf16(x, s);
}

// ---------------------------------------------------------- host helpers ---
void set_error(const char* fmt, ...);
nvfp4_status fail(nvfp4_status st, const char* fmt, ...);
nvfp4_status check_cuda(cudaError_t e, const char* what);

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Device address of the current device's status word (kernels record a
// nonzero nvfp4_status there instead of trapping); nullptr on failure.
int* device_status_ptr();

// Multiprocessor count of the current device (cached per device).
int sm_count();

// The dense GEMM behind nvfp4_w4a16_gemm / nvfp4_w4a16_gemm_f16 (argument
// checks, then the decode or the tile kernel), for layers built from it.
nvfp4_status run_dense_gemm(const void* X, const void* repacked, const void* pre_quant_scale, int64_t M,
                            int64_t N, int64_t K, void* Y, void* workspace, size_t workspace_bytes, bool f16,
                            void* stream);

// Kernels record the first error only.
__device__ __forceinline__ void record_status(int* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

}  // namespace nvfp4
