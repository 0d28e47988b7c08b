// One-time repack of a checkpoint-layout NVFP4 weight into the tiled layout,
// and the standalone dequant of a repacked weight to BF16.
//
// Format sources: "[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt on
// Hopper" (Changes table: E2M1 codebook lookup, per-block FP8 scale, per-tensor
// scale; the packed weight is K-packed innermost and the linear scale is
// row-major), SGLang PR 40022 (Motivation: gs=16 with E4M3 group scales;
// "Note the global-scale inversion": the divisor form is inverted before use).
// The repack plays the role of the pages' load-time Marlin repack / derived
// scale buffer: a pure function of its inputs.
#include "common.cuh"

namespace nvfp4 {
namespace {

// E4M3 (float8_e4m3fn) code -> value, from its fields.  NaN for 0x7F/0xFF.
__device__ double e4m3_to_double(uint32_t c) {
    const uint32_t e = (c >> 3) & 0xF, m = c & 7;
    double mag;
    if (e == 15 && m == 7) {
        mag = __longlong_as_double(0x7FF8000000000000ll);
    } else if (e == 0) {
        mag = ldexp((double)m, -9);                 // m/8 * 2^-6
    } else {
        mag = ldexp((double)(8 + m), (int)e - 10);  // (1 + m/8) * 2^(e-7)
    }
    return (c & 0x80) ? -mag : mag;
}

// Round a double to BF16, nearest-even, on the bit pattern: keep the top 7 of
// the 52 fraction bits (round at bit 45) for normal results, use the fixed
// 2^-133 grid for BF16 subnormals, overflow to infinity.
__device__ uint16_t bf16_from_double(double v) {
    const unsigned long long b = (unsigned long long)__double_as_longlong(v);
    const uint16_t sign = (uint16_t)((b >> 48) & 0x8000);
    const unsigned long long a = b & 0x7FFFFFFFFFFFFFFFull;
    if (a > 0x7FF0000000000000ull) return sign | 0x7FC0;   // NaN
    if (a == 0x7FF0000000000000ull) return sign | 0x7F80;  // inf
    const double x = __longlong_as_double((long long)a);
    if (x < 0x1p-126) {
        const double q = rint(x * 0x1p133);                  // exact scaling, RNE
        return sign | (uint16_t)q;                           // 128 -> min normal
    }
    const unsigned long long lsb = (a >> 45) & 1ull;
    unsigned long long r = a + 0x0FFFFFFFFFFFull + lsb;      // + (2^44 - 1) + lsb
    r &= ~((1ull << 45) - 1ull);
    const int e = (int)(r >> 52) - 1023 + 127;
    if (e >= 255) return sign | 0x7F80;
    return sign | (uint16_t)(e << 7) | (uint16_t)((r >> 45) & 0x7F);
}

// Round a double to FP16 (IEEE binary16), nearest-even, on the bit pattern:
// keep the top 10 of the 52 fraction bits (round at bit 42) for normal
// results, use the fixed 2^-24 grid for FP16 subnormals, overflow to infinity.
__device__ uint16_t f16_from_double(double v) {
    const unsigned long long b = (unsigned long long)__double_as_longlong(v);
    const uint16_t sign = (uint16_t)((b >> 48) & 0x8000);
    const unsigned long long a = b & 0x7FFFFFFFFFFFFFFFull;
    if (a > 0x7FF0000000000000ull) return sign | 0x7E00;   // NaN
    if (a == 0x7FF0000000000000ull) return sign | 0x7C00;  // inf
    const double x = __longlong_as_double((long long)a);
    if (x < 0x1p-14) {
        const double q = rint(x * 0x1p24);                   // exact scaling, RNE
        return sign | (uint16_t)q;                           // 1024 -> min normal
    }
    const unsigned long long lsb = (a >> 42) & 1ull;
    unsigned long long r = a + 0x1FFFFFFFFFFull + lsb;       // + (2^41 - 1) + lsb
    r &= ~((1ull << 42) - 1ull);
    const int e = (int)(r >> 52) - 1023 + 15;
    if (e >= 31) return sign | 0x7C00;
    return sign | (uint16_t)(e << 10) | (uint16_t)((r >> 42) & 0x3FF);
}

// Magnitude tables: entry s holds RN(mag_j * e4m3(s) * g) for the eight E2M1
// magnitudes j, once rounded to BF16 and once to FP16 (the two activation
// types).  The product is exact in double (<= 30 significant bits), so each
// entry is rounded exactly once.
__global__ void lut_kernel(uint8_t* out, float g, int64_t N, int64_t K, int64_t Np, int64_t Kp,
                           float global_scale, uint32_t is_div) {
    const int s = threadIdx.x;          // 256 threads
    const double mags[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    const double sv = e4m3_to_double((uint32_t)s);
    // sign of a NaN weight = sign(scale) xor sign(g) (code sign applied later)
    const uint16_t nan_sign = (uint16_t)((((uint32_t)s >> 7) ^ (__float_as_uint(g) >> 31)) << 15);
    uint8_t lo[2][8], hi[2][8];
    for (int j = 0; j < 8; ++j) {
        const double v = mags[j] * sv * (double)g;
        uint16_t bits[2] = {bf16_from_double(v), f16_from_double(v)};
        if (isnan(v)) {
            bits[0] = (uint16_t)(0x7FC0 | nan_sign);
            bits[1] = (uint16_t)(0x7E00 | nan_sign);
        }
        for (int t = 0; t < 2; ++t) {
            lo[t][j] = (uint8_t)(bits[t] & 0xFF);
            hi[t][j] = (uint8_t)(bits[t] >> 8);
        }
    }
    for (int t = 0; t < 2; ++t) {
        uint8_t* e = out + (t ? kLutF16Offset : kLutBf16Offset) + (size_t)s * 16;
        for (int j = 0; j < 8; ++j) { e[j] = lo[t][j]; e[8 + j] = hi[t][j]; }
    }
    if (s == 0) {
        Header h{};
        h.magic = kMagic; h.version = kVersion;
        h.N = N; h.K = K; h.Np = Np; h.Kp = Kp;
        h.g = g; h.global_scale = global_scale; h.global_is_divisor = is_div;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(&h);
        for (int i = 0; i < (int)sizeof(Header); ++i) out[i] = src[i];
        for (int i = (int)sizeof(Header); i < (int)kHeaderBytes; ++i) out[i] = 0;
    }
}

// Natural order word (nibble i = code of element i) -> sign-split word.
__device__ __forceinline__ uint32_t to_sign_split(uint32_t w) {
    const int sign_pos[8] = {7, 15, 23, 31, 3, 11, 19, 27};
    uint32_t out = w & 0x77777777u;
    #pragma unroll
    for (int i = 0; i < 8; ++i) out |= ((w >> (4 * i + 3)) & 1u) << sign_pos[i];
    return out;
}

// Byte offset of the scale of row n, 16-group j in the swizzled checkpoint
// layout (G groups per row): 128-row x 4-group tiles of 512 bytes, row-tile
// major, and inside a tile (r % 32) * 16 + (r / 32) * 4 + (j % 4), r = n % 128.
__device__ __forceinline__ int64_t swizzled_scale_offset(int64_t n, int64_t j, int64_t G) {
    const int64_t tile = (n / 128) * ((G + 3) / 4) + j / 4;
    const int64_t r = n % 128;
    return tile * 512 + (r % 32) * 16 + (r / 32) * 4 + (j % 4);
}

// One warp per atom.  Lane L = 4r + q writes its 16 code bytes (rows r, r+8 of
// the atom, group q) and its 2 scale bytes.
__global__ void tiles_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                             uint8_t* __restrict__ out, int64_t N, int64_t K, int64_t KB,
                             int64_t total_atoms, int swizzled) {
    const int64_t atom = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (atom >= total_atoms) return;
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2, q = lane & 3;
    const int64_t rb = atom % kAtomsPerTileK;
    const int64_t kb = (atom / kAtomsPerTileK) % KB;
    const int64_t nt = atom / (kAtomsPerTileK * KB);
    const int64_t k0 = kb * kBlockK + q * kGroup;
    uint32_t words[4];
    uint8_t sc[2];
    for (int h = 0; h < 2; ++h) {
        const int64_t n = nt * kTileRows + rb * kAtomRows + r + 8 * h;
        uint2 raw = make_uint2(0u, 0u);
        uint8_t s = 0;
        if (n < N && k0 < K) {
            raw = *reinterpret_cast<const uint2*>(packed + n * (K / 2) + k0 / 2);
            const int64_t G = K / kGroup, j = k0 / kGroup;
            s = swizzled ? scales[swizzled_scale_offset(n, j, G)] : scales[n * G + j];
        }
        words[2 * h] = to_sign_split(raw.x);
        words[2 * h + 1] = to_sign_split(raw.y);
        sc[h] = s;
    }
    uint8_t* a = out + kTilesOffset + (size_t)atom * kAtomBytes;
    *reinterpret_cast<uint4*>(a + 16 * lane) = make_uint4(words[0], words[1], words[2], words[3]);
    a[kAtomCodeBytes + 2 * lane] = sc[0];
    a[kAtomCodeBytes + 2 * lane + 1] = sc[1];
}

// Standalone dequant: one warp per atom, each lane expands its 32 elements
// through the magnitude table of the activation type (the same expansion the
// GEMM kernels use) and stores the valid ones.
template <bool F16>
__global__ void dequant_kernel(const uint8_t* __restrict__ rp, uint16_t* __restrict__ out,
                               int64_t N, int64_t K, int64_t KB, int64_t total_atoms, int* status) {
    __shared__ uint4 lut[256];
    const Header* hdr = reinterpret_cast<const Header*>(rp);
    if (hdr->magic != kMagic || hdr->N != N || hdr->K != K) {
        if (threadIdx.x == 0 && blockIdx.x == 0) record_status(status, NVFP4_ERR_BAD_WEIGHT);
        return;
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        lut[i] = reinterpret_cast<const uint4*>(rp + lut_offset<F16>())[i];
    __syncthreads();
    const int64_t atom = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (atom >= total_atoms) return;
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2, q = lane & 3;
    const int64_t rb = atom % kAtomsPerTileK;
    const int64_t kb = (atom / kAtomsPerTileK) % KB;
    const int64_t nt = atom / (kAtomsPerTileK * KB);
    const int64_t k0 = kb * kBlockK + q * kGroup;
    const uint8_t* a = rp + kTilesOffset + (size_t)atom * kAtomBytes;
    const uint4 codes = *reinterpret_cast<const uint4*>(a + 16 * lane);
    const uint8_t s0 = a[kAtomCodeBytes + 2 * lane], s1 = a[kAtomCodeBytes + 2 * lane + 1];
    const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
    for (int h = 0; h < 2; ++h) {
        const int64_t n = nt * kTileRows + rb * kAtomRows + r + 8 * h;
        if (n >= N || k0 >= K) continue;
        const Lut t = lut_from_uint4(lut[h ? s1 : s0]);
        uint32_t e[8];
        expand8(w[2 * h], t, e);
        expand8(w[2 * h + 1], t, e + 4);
        uint4* dst = reinterpret_cast<uint4*>(out + n * K + k0);
        dst[0] = make_uint4(e[0], e[1], e[2], e[3]);
        dst[1] = make_uint4(e[4], e[5], e[6], e[7]);
    }
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" size_t nvfp4_repack_size(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % kGroup != 0) return 0;
    const int64_t Np = round_up(N, kTileRows), Kp = round_up(K, kBlockK);
    const size_t atoms = (size_t)(Np / kAtomRows) * (size_t)(Kp / kBlockK);
    return (size_t)round_up((int64_t)(kTilesOffset + atoms * kAtomBytes), 256);
}

extern "C" size_t nvfp4_swizzled_scales_size(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % kGroup != 0) return 0;
    return (size_t)(round_up(N, 128) * round_up(K / kGroup, 4));
}

extern "C" nvfp4_status nvfp4_repack_ex(const uint8_t* packed, const uint8_t* scales_e4m3, int scale_layout,
                                        float global_scale, int global_is_divisor,
                                        int64_t N, int64_t K, void* out, size_t out_bytes,
                                        void* stream) {
    const char* fn = scale_layout == NVFP4_SCALES_LINEAR ? "nvfp4_repack" : "nvfp4_repack_ex";
    if (scale_layout != NVFP4_SCALES_LINEAR && scale_layout != NVFP4_SCALES_SWIZZLED_128x4)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: scale_layout=%d is not LINEAR or SWIZZLED_128x4", fn, scale_layout);
    if (N <= 0 || K <= 0) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: N=%lld K=%lld must be positive", fn, (long long)N, (long long)K);
    if (K % kGroup != 0) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: K=%lld is not a multiple of the group size 16", fn, (long long)K);
    if (!packed || !scales_e4m3 || !out) return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer (packed=%p scales=%p out=%p)", fn, (const void*)packed, (const void*)scales_e4m3, out);
    if (global_is_divisor != 0 && global_is_divisor != 1) return fail(NVFP4_ERR_INVALID_ARG, "%s: global_is_divisor must be 0 or 1", fn);
    if (!aligned(packed, 16)) return fail(NVFP4_ERR_ALIGNMENT, "%s: packed weight must be 16-byte aligned", fn);
    if (!aligned(out, 256)) return fail(NVFP4_ERR_ALIGNMENT, "%s: out must be 256-byte aligned", fn);
    const size_t need = nvfp4_repack_size(N, K);
    if (out_bytes < need) return fail(NVFP4_ERR_WORKSPACE, "%s: out has %zu bytes, needs %zu", fn, out_bytes, need);
    // g = RN_fp32(1/d): one IEEE single-precision division.
    volatile float one = 1.0f;
    const float g = global_is_divisor ? one / global_scale : global_scale;
    if (!(g == g) || g == 0.0f || g == INFINITY || g == -INFINITY)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: global multiplier %g (from %g, divisor=%d) must be finite and nonzero", fn, (double)g, (double)global_scale, global_is_divisor);
    const int64_t Np = round_up(N, kTileRows), Kp = round_up(K, kBlockK);
    const int64_t KB = Kp / kBlockK;
    const int64_t atoms = (Np / kAtomRows) * KB;
    cudaStream_t s = (cudaStream_t)stream;
    lut_kernel<<<1, 256, 0, s>>>((uint8_t*)out, g, N, K, Np, Kp, global_scale, (uint32_t)global_is_divisor);
    nvfp4_status st = check_cuda(cudaGetLastError(), "nvfp4_repack: magnitude-table launch");
    if (st != NVFP4_OK) return st;
    const int warps = 8;
    tiles_kernel<<<(unsigned)ceil_div(atoms, warps), warps * 32, 0, s>>>(packed, scales_e4m3, (uint8_t*)out, N, K, KB,
                                                                         atoms, scale_layout);
    return check_cuda(cudaGetLastError(), "nvfp4_repack: tile launch");
}

extern "C" nvfp4_status nvfp4_repack(const uint8_t* packed, const uint8_t* scales_e4m3,
                                     float global_scale, int global_is_divisor,
                                     int64_t N, int64_t K, void* out, size_t out_bytes,
                                     void* stream) {
    return nvfp4_repack_ex(packed, scales_e4m3, NVFP4_SCALES_LINEAR, global_scale, global_is_divisor, N, K, out,
                           out_bytes, stream);
}

namespace nvfp4 {
namespace {

nvfp4_status dequant_impl(const void* repacked, int64_t N, int64_t K, uint16_t* out, bool f16, void* stream) {
    const char* fn = f16 ? "nvfp4_dequant_f16" : "nvfp4_dequant";
    if (N <= 0 || K <= 0 || K % kGroup != 0) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: N=%lld K=%lld (K must be a positive multiple of 16)", fn, (long long)N, (long long)K);
    if (!repacked || !out) return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(repacked, 256)) return fail(NVFP4_ERR_ALIGNMENT, "%s: repacked weight must be 256-byte aligned", fn);
    if (!aligned(out, 16)) return fail(NVFP4_ERR_ALIGNMENT, "%s: out must be 16-byte aligned", fn);
    const int64_t Np = round_up(N, kTileRows), KB = round_up(K, kBlockK) / kBlockK;
    const int64_t atoms = (Np / kAtomRows) * KB;
    int* status = device_status_ptr();
    if (!status) return fail(NVFP4_ERR_CUDA, "%s: no CUDA device", fn);
    const int warps = 8;
    const unsigned grid = (unsigned)ceil_div(atoms, warps);
    if (f16)
        dequant_kernel<true><<<grid, warps * 32, 0, (cudaStream_t)stream>>>((const uint8_t*)repacked, out, N, K, KB, atoms, status);
    else
        dequant_kernel<false><<<grid, warps * 32, 0, (cudaStream_t)stream>>>((const uint8_t*)repacked, out, N, K, KB, atoms, status);
    return check_cuda(cudaGetLastError(), f16 ? "nvfp4_dequant_f16: launch" : "nvfp4_dequant: launch");
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_dequant(const void* repacked, int64_t N, int64_t K,
                                      uint16_t* out_bf16, void* stream) {
    return dequant_impl(repacked, N, K, out_bf16, false, stream);
}

extern "C" nvfp4_status nvfp4_dequant_f16(const void* repacked, int64_t N, int64_t K,
                                          uint16_t* out_f16, void* stream) {
    return dequant_impl(repacked, N, K, out_f16, true, stream);
}
