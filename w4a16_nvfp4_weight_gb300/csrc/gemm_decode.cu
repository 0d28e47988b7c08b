// Decode-shaped W4A16 GEMM (few tokens): split-K, HBM-streaming, with the
// dequant fused into the tensor-core operand registers.
//
// The weight is the only large operand, so every byte of it is read once with
// 128-bit streaming loads.  Each warp owns 16 weight rows; per 64-k atom a lane
// loads 16 code bytes and 2 scale bytes, looks its two group tables up in
// shared memory and expands the codes straight into mma.sync A fragments
// (weights on the M side, tokens on the N side).  Within a 16-element group
// the MMA's k order is permuted so that one lane consumes one whole group of
// one row per four MMAs; the activation fragments follow the same permutation,
// so the dot products are unchanged.  K is split across the CTAs of a thread
// block cluster, which reduce their FP32 partials through distributed shared
// memory in rank order: deterministic, and no global workspace.
//
// Method: "[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt on Hopper"
// (Description / Changes table: dequantize the NVFP4 weight each forward step
// and run a BF16 GEMM); AWQ activation scaling from "[None][fix] Apply the
// NVFP4_AWQ pre-quant scale in MegaMoE CuteDSL" (Description).
#include <cooperative_groups.h>

#include "common.cuh"
#include "gemm_decode.cuh"

namespace cg = cooperative_groups;

namespace nvfp4 {

__device__ __forceinline__ void mma_bf16_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

namespace {

constexpr int kWarps = 8;                     // 8 x 16 = 128 weight rows per CTA
constexpr int kRowsPerCta = kWarps * kAtomRows;
constexpr int kUnroll = 4;                    // atoms in flight per warp

// Process one atom held in registers: expand and issue 4 x MT MMAs.
template <int MT>
__device__ __forceinline__ void atom_mma(const uint4 codes, uint32_t sc2, const uint4* lut,
                                         const uint16_t* xs, int x_stride, int kl, int lane,
                                         float acc[MT][4]) {
    const Lut t0 = lut_from_uint4(lut[sc2 & 0xFF]);
    const Lut t1 = lut_from_uint4(lut[(sc2 >> 8) & 0xFF]);
    uint32_t ra[8], rb[8];
    expand8(codes.x, t0, ra);
    expand8(codes.y, t0, ra + 4);
    expand8(codes.z, t1, rb);
    expand8(codes.w, t1, rb + 4);
    const int g = lane >> 2, q = lane & 3;
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t a[4] = {ra[2 * j], rb[2 * j], ra[2 * j + 1], rb[2 * j + 1]};
        #pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const uint2 b = *reinterpret_cast<const uint2*>(xs + (mt * 8 + g) * x_stride + kl + q * 16 + 4 * j);
            mma_bf16_16816(acc[mt], a, b.x, b.y);
        }
    }
}

template <int MT>
__global__ void __launch_bounds__(kWarps * 32)
decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint4* lut = reinterpret_cast<uint4*>(smem);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + kLutBytes);
    float* part = reinterpret_cast<float*>(smem + kLutBytes + (size_t)MT * 8 * p.x_stride * 2);
    constexpr int TOK = 8 * MT;

    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = blockIdx.x;
    const int split = blockIdx.y;
    const int64_t m0 = (int64_t)blockIdx.z * TOK;

    // Every CTA reads the same header, so all CTAs of a cluster agree.
    const Header* hdr = reinterpret_cast<const Header*>(p.rp);
    if (hdr->magic != kMagic || hdr->N != p.N || hdr->K != p.K) {
        if (tid == 0) record_status(p.status, NVFP4_ERR_BAD_WEIGHT);
        return;
    }

    for (int i = tid; i < 256; i += blockDim.x)
        lut[i] = reinterpret_cast<const uint4*>(p.rp + kHeaderBytes)[i];

    const int kb0 = split * p.kbs;
    const int kb1 = min(kb0 + p.kbs, (int)p.KB);
    const int nk = (kb1 - kb0) * kBlockK;           // local k extent
    // Stage this split's activation slice (zero beyond M and K), applying the
    // AWQ pre-quant scale when present.
    const int chunks = nk / 8;
    for (int i = tid; i < TOK * chunks; i += blockDim.x) {
        const int t = i / chunks, c = i % chunks;
        const int64_t m = m0 + t;
        const int64_t k = (int64_t)kb0 * kBlockK + c * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (m < p.M && k < p.K) {
            v = *reinterpret_cast<const uint4*>(p.X + m * p.K + k);
            if (p.pqs != nullptr) {
                const uint4 s = *reinterpret_cast<const uint4*>(p.pqs + k);
                uint32_t xv[4] = {v.x, v.y, v.z, v.w};
                const uint32_t sv[4] = {s.x, s.y, s.z, s.w};
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint16_t lo = awq_mul_bf16((uint16_t)(xv[e] & 0xFFFF), (uint16_t)(sv[e] & 0xFFFF));
                    const uint16_t hi = awq_mul_bf16((uint16_t)(xv[e] >> 16), (uint16_t)(sv[e] >> 16));
                    xv[e] = (uint32_t)lo | ((uint32_t)hi << 16);
                }
                v = make_uint4(xv[0], xv[1], xv[2], xv[3]);
            }
        }
        uint16_t* dst = xs + t * p.x_stride + c * 8;
        // x_stride is a multiple of 4 elements: 8-byte aligned rows
        reinterpret_cast<uint2*>(dst)[0] = make_uint2(v.x, v.y);
        reinterpret_cast<uint2*>(dst)[1] = make_uint2(v.z, v.w);
    }
    __syncthreads();

    float acc[MT][4];
    #pragma unroll
    for (int mt = 0; mt < MT; ++mt)
        #pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.0f;

    const int64_t rbg = (int64_t)rg * kWarps + warp;          // global 16-row block
    if (rbg * kAtomRows < p.N) {
        const int64_t nt = rbg / kAtomsPerTileK, rb = rbg % kAtomsPerTileK;
        const uint8_t* tiles = p.rp + kTilesOffset;
        const size_t kb_stride = (size_t)kAtomsPerTileK * kAtomBytes;
        const uint8_t* a0 = tiles + atom_offset(nt, kb0, rb, p.KB);
        int kb = kb0;
        for (; kb + kUnroll <= kb1; kb += kUnroll) {
            uint4 c[kUnroll];
            uint32_t s[kUnroll];
            #pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint8_t* a = a0 + (size_t)(kb - kb0 + u) * kb_stride;
                c[u] = ldg_stream(a + 16 * lane);
                s[u] = ldg_u16(a + kAtomCodeBytes + 2 * lane);
            }
            #pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                atom_mma<MT>(c[u], s[u], lut, xs, p.x_stride, (kb - kb0 + u) * kBlockK, lane, acc);
        }
        for (; kb < kb1; ++kb) {
            const uint8_t* a = a0 + (size_t)(kb - kb0) * kb_stride;
            const uint4 c = ldg_stream(a + 16 * lane);
            const uint32_t s = ldg_u16(a + kAtomCodeBytes + 2 * lane);
            atom_mma<MT>(c, s, lut, xs, p.x_stride, (kb - kb0) * kBlockK, lane, acc);
        }
    }

    // Partials: part[row][token], row = warp*16 + (g or g+8), token = mt*8 + 2c (+1)
    {
        const int g = lane >> 2, c = lane & 3;
        #pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            float* r0 = part + (warp * 16 + g) * TOK + mt * 8 + 2 * c;
            float* r8 = part + (warp * 16 + g + 8) * TOK + mt * 8 + 2 * c;
            r0[0] = acc[mt][0]; r0[1] = acc[mt][1];
            r8[0] = acc[mt][2]; r8[1] = acc[mt][3];
        }
    }
    cluster.sync();

    // Each CTA of the cluster reduces a contiguous share of the outputs, summing
    // the partials of ranks 0..splits-1 in order.
    const int total = kRowsPerCta * TOK;
    const int splits = p.splits;
    const int share = (total + splits - 1) / splits;
    const int e0 = split * share, e1 = min(total, e0 + share);
    for (int e = e0 + tid; e < e1; e += blockDim.x) {
        const int t = e / kRowsPerCta, row = e % kRowsPerCta;      // consecutive e -> consecutive n
        float sum = 0.0f;
        for (int r = 0; r < splits; ++r) {
            const float* peer = cluster.map_shared_rank(part, r);
            sum += peer[row * TOK + t];
        }
        const int64_t n = (int64_t)rg * kRowsPerCta + row;
        const int64_t m = m0 + t;
        if (n < p.N && m < p.M) p.Y[m * p.N + n] = f32_to_bf16_bits(sum);
    }
    cluster.sync();   // keep this CTA's partials alive until every peer has read them
}

}  // namespace

size_t decode_smem_bytes(int MT, int kbs) {
    const int x_stride = kbs * kBlockK + 4;
    return kLutBytes + (size_t)MT * 8 * x_stride * 2 + (size_t)kRowsPerCta * MT * 8 * 4;
}

nvfp4_status launch_decode(const DecodeParams& p_in, int MT, cudaStream_t stream) {
    DecodeParams p = p_in;
    p.x_stride = p.kbs * kBlockK + 4;
    const size_t smem = decode_smem_bytes(MT, p.kbs);
    const void* fn = MT == 1 ? (const void*)decode_kernel<1> : (const void*)decode_kernel<2>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return check_cuda(e, "decode GEMM: shared memory attribute");
    const int64_t rgs = ceil_div(p.N, kRowsPerCta);
    const int64_t mchunks = ceil_div(p.M, 8 * MT);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rgs, (unsigned)p.splits, (unsigned)mchunks);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)p.splits;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (MT == 1) e = cudaLaunchKernelEx(&cfg, decode_kernel<1>, p);
    else e = cudaLaunchKernelEx(&cfg, decode_kernel<2>, p);
    return check_cuda(e, "decode GEMM: launch");
}

}  // namespace nvfp4
