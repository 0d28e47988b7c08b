// Tensor-core tile GEMMs for the W4A16 NVFP4 linear at larger M (prefill, LM
// head, MoE with many rows per expert): dequant-fused, TMA-fed, tcgen05 MMAs
// accumulating in tensor memory.  Two kernels: tc_gemm_kernel (below; both
// operands in shared memory; dense and the MoE / MLP epilogues) and
// tc_wa_kernel (further down; dense only; the dequantized weights as the
// tensor-memory A operand).  plan_tc picks one per dense shape.
//
// tc_gemm_kernel: one CTA computes a (128*SUBM) x 256 output tile over its K range:
//   warp 0      producer: per 64-k block, TMA tile loads of the activation
//               (128 rows x 64 k, 128-byte swizzle, zero fill past M and K)
//               and one bulk copy of the weight block (256 rows x 64 k of codes
//               and scales, 9216 contiguous bytes) into a 3-stage ring;
//   warp 1      allocates 256*SUBM tensor-memory columns and issues, per block,
//               SUBM x 4 tcgen05 BF16 MMAs (M=128, N=256, K=16) from shared
//               memory into the FP32 accumulators; commits release the stages;
//   warps 2..9  expand the weight codes through the magnitude table into the
//               BF16 B operand (256 x 64, 128-byte swizzled K-major layout) of a
//               2-stage ring, then run the epilogue: tensor memory -> registers
//               -> BF16 -> global, rows/columns past M/N clipped.
// The weight tile is dequantized once per CTA and shared by the SUBM M
// sub-tiles, so the dequant (integer pipe) work per FLOP halves at SUBM = 2.
//
// Method: "[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt on Hopper"
// (Description / Changes table: NVFP4 weights dequantized per step, BF16 GEMM);
// AWQ: "[None][fix] Apply the NVFP4_AWQ pre-quant scale in MegaMoE CuteDSL"
// (the activation is scaled in BF16 before the GEMM; done by a pre-pass here).
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "gemm_decode.cuh"
#include "gemm_tc.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kTcThreads = 320;                  // 10 warps
constexpr int kDeqWarps = 8;
constexpr int kS1 = 3;                           // activation + raw-weight ring
constexpr int kS2 = 2;                           // dequantized-weight ring
constexpr int kBN = 256;
constexpr uint32_t kATileBytes = 128 * 64 * 2;   // 16 KB per 128-row sub-tile
constexpr uint32_t kBRawBytes = kAtomsPerTileK * kAtomBytes;   // 9216
constexpr uint32_t kBDeqBytes = kBN * 64 * 2;    // 32 KB

template <int SUBM>
struct TcSmem {
    static constexpr size_t a = 0;                                            // 1024-aligned
    static constexpr size_t bdeq = a + (size_t)kS1 * SUBM * kATileBytes;      // 1024-aligned
    static constexpr size_t braw = bdeq + (size_t)kS2 * kBDeqBytes;
    static constexpr size_t lut = braw + (size_t)kS1 * kBRawBytes;          // + a second table
    static constexpr size_t bars = lut + 2 * kLutBytes;                      //   for gate/up shards
    static constexpr size_t misc = bars + 16 * 8;
    static constexpr size_t total = misc + 64;
};

// kMoeFc1: gated FC1 (gate/up + SwiGLU -> H); kMoeFc1Plain: non-gated FC1
// (relu2 or silu -> H); kMoeFc2: x p -> FP32 rows per routing slot.
enum class TcMode { kDense, kMoeFc1, kMoeFc1Plain, kMoeFc2 };

struct TcKParams {
    const uint8_t* rp;        // dense: the repacked weight; MoE: expert 0 of the stacked weights
    size_t w_stride;          // MoE: bytes between experts
    uint16_t* Y;              // dense: [M, N] BF16; MoE FC1: H [rows, I] BF16
    float* Yp;                // MoE FC2: [slots, N] FP32, scaled by the routing weight
    const int4* items;        // MoE: (expert, first row, rows, -) work list; null with one
                              //   dense weight: runs of 128*SUBM rows of M
    const int32_t* n_items;
    const int32_t* perm;      // MoE FC2: permuted row -> routing slot
    const float* wts;         // MoE FC2: routing weights per slot
    int64_t M, N, K, KB;      // dense M; weight rows N (FC1: 2I) and inner K
    int64_t I;                // MoE FC1: intermediate size
    size_t half_stride;       // gated FC1: 0 = one [2I, K] weight, else bytes from the gate
                              //   shard [I, K] to the up shard [I, K] (own globals)
    int act;                  // non-gated FC1: 1 = relu2, 2 = silu
    int kb_per_split;         // dense split-K: 64-k blocks per split (grid z = split)
    float* partial;           // dense split-K: FP32 partials [splits, M, N], or null
    int* status;
};

// Byte offset of the 16-byte chunk c (0..7) of row n in a 128-byte swizzled
// K-major tile.
__device__ __forceinline__ uint32_t sw128_offset(int n, int c) {
    return (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((c ^ (n & 7)) << 4));
}

__device__ __forceinline__ float silu_tc(float v) { return v / (1.0f + expf(-v)); }

__device__ __forceinline__ float plain_act_tc(float v, int act) {
    if (act == 1) {
        const float r = fmaxf(v, 0.0f);
        return r * r;
    }
    return silu_tc(v);
}

// Warp-cooperative store of a block of 32 rows x 32 words: lane l holds the 32
// consecutive 32-bit words of row l, bound for dst (16-byte aligned; null: row l
// is not stored); only the first `valid` words of each row are stored (a
// multiple of 4, the same for the whole warp).  The rows pass through a
// 32 x 33-word tile in shared memory so that each 16-byte store belongs to a run
// of 8 lanes writing 128 contiguous bytes of one row -- four rows per store
// instruction instead of 16 bytes of each of 32 rows.
__device__ __forceinline__ void store_rows32(uint32_t* tile, const uint32_t (&w)[32], uint32_t* dst, int valid,
                                             int lane) {
    #pragma unroll
    for (int i = 0; i < 32; ++i) tile[lane * 33 + i] = w[i];
    __syncwarp();
    const int c = (lane & 7) * 4;
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = i * 4 + (lane >> 3);
        uint32_t* d = reinterpret_cast<uint32_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst), r));
        const uint32_t* s = tile + r * 33 + c;
        if (d != nullptr && c < valid) *reinterpret_cast<uint4*>(d + c) = make_uint4(s[0], s[1], s[2], s[3]);
    }
    __syncwarp();
}

__device__ __forceinline__ uint32_t pack_act2(uint32_t a, uint32_t b, bool f16) {
    return f16 ? ((uint32_t)f32_to_act_bits<true>(__uint_as_float(a)) |
                  ((uint32_t)f32_to_act_bits<true>(__uint_as_float(b)) << 16))
               : ((uint32_t)f32_to_act_bits<false>(__uint_as_float(a)) |
                  ((uint32_t)f32_to_act_bits<false>(__uint_as_float(b)) << 16));
}

template <int SUBM, TcMode MODE, bool F16>
__global__ void __launch_bounds__(kTcThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const TcKParams p) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled operand tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = TcSmem<SUBM>;
    uint8_t* a_ring = smem + L::a;
    uint8_t* bdeq_ring = smem + L::bdeq;
    uint8_t* braw_ring = smem + L::braw;
    uint4* lut = reinterpret_cast<uint4*>(smem + L::lut);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
    uint64_t* tma_full = bars;                    // [kS1]
    uint64_t* tma_empty = bars + kS1;             // [kS1]
    uint64_t* deq_full = bars + 2 * kS1;          // [kS2]
    uint64_t* deq_empty = bars + 2 * kS1 + kS2;   // [kS2]
    uint64_t* acc_full = bars + 2 * kS1 + 2 * kS2;
    uint64_t* lut_bar = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc);
    volatile int* hdr_flag = reinterpret_cast<volatile int*>(smem + L::misc + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr bool kMoe = MODE != TcMode::kDense;
    // dense: output tile (m0, n0); MoE: work item (expert, first permuted row,
    // rows) and output columns n0 (FC1: intermediate columns j0 = 128 * bx)
    int64_t m0, m_end;
    const uint8_t* wbase = p.rp;
    if constexpr (kMoe) {
        int4 item;                                      // uniform across the CTA
        if (p.items != nullptr) {
            if ((int)blockIdx.y >= *p.n_items) return;
            item = p.items[blockIdx.y];
        } else {
            // one dense weight (FC1 of a dense MLP): consecutive runs of token rows
            const int64_t first = (int64_t)blockIdx.y * 128 * SUBM;
            if (first >= p.M) return;
            item = make_int4(0, (int)first, (int)(p.M - first < 128 * SUBM ? p.M - first : 128 * SUBM), 0);
        }
        wbase = p.rp + (size_t)item.x * p.w_stride;
        m0 = item.y;
        m_end = (int64_t)item.y + item.z;
    } else {
        m0 = (int64_t)blockIdx.y * 128 * SUBM;
        m_end = p.M;
    }
    const int64_t n0 = (int64_t)blockIdx.x * (MODE == TcMode::kMoeFc1 ? kBN / 2 : kBN);
    const bool shards = MODE == TcMode::kMoeFc1 && p.half_stride != 0;
    const uint8_t* wbase_up = shards ? wbase + p.half_stride : wbase;
    // dense split-K: this CTA covers 64-k blocks [kb_first, kb_first + nkb)
    const int kb_first = kMoe ? 0 : (int)blockIdx.z * p.kb_per_split;
    const int64_t kb_left = p.KB - kb_first;
    const int nkb = kMoe ? (int)p.KB : (int)(kb_left < p.kb_per_split ? kb_left : p.kb_per_split);

    if (tid == 0) {
        for (int s = 0; s < kS1; ++s) {
            mbar_init(&tma_full[s], 1);
            mbar_init(&tma_empty[s], 1 + kDeqWarps);   // MMA commit + every dequant warp
        }
        for (int s = 0; s < kS2; ++s) {
            mbar_init(&deq_full[s], kDeqWarps);
            mbar_init(&deq_empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(lut_bar, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 256 * SUBM);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // A kernel launched after this one with programmatic dependent launch may
    // start now (its CTAs fill SMs as this grid's last wave drains); it waits
    // for this kernel (griddepcontrol.wait) before it reads what this writes.
    // Launches of the tile kernels themselves are ordinary stream launches.
    if (tid == 0) pdl_launch_dependents();
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t idesc = umma_idesc(128, kBN, F16);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const Header* hdr = reinterpret_cast<const Header*>(wbase);
            const Header* hdr_up = reinterpret_cast<const Header*>(wbase_up);
            const bool ok_hdr = hdr->magic == kMagic && hdr->N == p.N && hdr->K == p.K &&
                                (!shards || (hdr_up->magic == kMagic && hdr_up->N == p.N && hdr_up->K == p.K));
            *hdr_flag = ok_hdr ? 1 : 0;
            if (!ok_hdr) {
                record_status(p.status, NVFP4_ERR_BAD_WEIGHT);
                mbar_arrive(lut_bar);
            } else {
                mbar_arrive_expect_tx(lut_bar, (uint32_t)((shards ? 2 : 1) * kLutBytes));
                bulk_g2s(lut, wbase + lut_offset<F16>(), (uint32_t)kLutBytes, lut_bar);
                if (shards) bulk_g2s(lut + 256, wbase_up + lut_offset<F16>(), (uint32_t)kLutBytes, lut_bar);
                // FC1: 128 gate rows j0.. and the 128 matching up rows (I + j0.. of the
                // same weight, or j0.. of the up shard): two half tiles; otherwise one
                // 256-row tile
                auto half_tile = [&](const uint8_t* base, int64_t row0) {
                    const int64_t rbg = row0 / kAtomRows;
                    return base + kTilesOffset + atom_offset(rbg / kAtomsPerTileK, 0, rbg % kAtomsPerTileK, p.KB);
                };
                const uint8_t* wtile = half_tile(wbase, n0);
                const uint8_t* wtile_up =
                    MODE == TcMode::kMoeFc1 ? half_tile(wbase_up, (shards ? 0 : p.I) + n0) : nullptr;
                int issued = 0;
                for (int kb = 0; kb < nkb; ++kb) {
                    const int s = kb % kS1;
                    if (kb >= kS1 && !mbar_wait(&tma_empty[s], ((kb / kS1) - 1) & 1, p.status)) break;
                    mbar_arrive_expect_tx(&tma_full[s], SUBM * kATileBytes + kBRawBytes);
                    for (int mi = 0; mi < SUBM; ++mi)
                        tma_load_2d(a_ring + ((size_t)s * SUBM + mi) * kATileBytes, &tmap_x, (kb_first + kb) * 64,
                                    (int)(m0 + mi * 128), &tma_full[s]);
                    if constexpr (MODE == TcMode::kMoeFc1) {
                        bulk_g2s(braw_ring + (size_t)s * kBRawBytes, wtile + (size_t)kb * kBRawBytes,
                                 kBRawBytes / 2, &tma_full[s]);
                        bulk_g2s(braw_ring + (size_t)s * kBRawBytes + kBRawBytes / 2,
                                 wtile_up + (size_t)kb * kBRawBytes, kBRawBytes / 2, &tma_full[s]);
                    } else {
                        bulk_g2s(braw_ring + (size_t)s * kBRawBytes, wtile + (size_t)(kb_first + kb) * kBRawBytes,
                                 kBRawBytes, &tma_full[s]);
                    }
                    ++issued;
                }
                // no copy may still target this CTA when it exits
                mbar_wait(lut_bar, 0, p.status);
                for (int kb = issued > kS1 ? issued - kS1 : 0; kb < issued; ++kb)
                    mbar_wait(&tma_full[kb % kS1], (kb / kS1) & 1, p.status);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            bool ok = mbar_wait(lut_bar, 0, p.status) && *hdr_flag != 0;
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s1 = kb % kS1, s2 = kb % kS2;
                ok = mbar_wait(&tma_full[s1], (kb / kS1) & 1, p.status) &&
                     mbar_wait(&deq_full[s2], (kb / kS2) & 1, p.status);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t a_base = smem_u32(a_ring + (size_t)s1 * SUBM * kATileBytes);
                const uint32_t b_base = smem_u32(bdeq_ring + (size_t)s2 * kBDeqBytes);
                #pragma unroll
                for (int mi = 0; mi < SUBM; ++mi)
                    #pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f16kind_ss(tmem + mi * kBN, sw128_kmajor_desc(a_base + mi * kATileBytes + kk * 32),
                                     sw128_kmajor_desc(b_base + kk * 32), idesc, (kb | kk) != 0);
                umma_commit(&tma_empty[s1]);
                umma_commit(&deq_empty[s2]);
            }
            umma_commit(acc_full);          // also waits out every MMA issued above
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ dequant, then epilogue
        const int dw = warp - 2;                        // 0..7: atoms 2dw, 2dw+1 of each block
        const int r = lane >> 2, q = lane & 3;
        const uint4* const dlut = (shards && dw >= 4) ? lut + 256 : lut;     // rows 128.. are up rows
        bool ok = mbar_wait(lut_bar, 0, p.status) && *hdr_flag != 0;
        for (int kb = 0; kb < nkb && ok; ++kb) {
            const int s1 = kb % kS1, s2 = kb % kS2;
            ok = mbar_wait(&tma_full[s1], (kb / kS1) & 1, p.status);
            if (ok && kb >= kS2) ok = mbar_wait(&deq_empty[s2], ((kb / kS2) - 1) & 1, p.status);
            if (!ok) break;
            const uint8_t* raw = braw_ring + (size_t)s1 * kBRawBytes;
            uint8_t* dst = bdeq_ring + (size_t)s2 * kBDeqBytes;
            #pragma unroll
            for (int ai = 0; ai < 2; ++ai) {
                const int atom = 2 * dw + ai;
                const uint8_t* a = raw + atom * kAtomBytes;
                const uint4 codes = *reinterpret_cast<const uint4*>(a + 16 * lane);
                const uint32_t sc2 = *reinterpret_cast<const uint16_t*>(a + kAtomCodeBytes + 2 * lane);
                const Lut t0 = lut_from_uint4(dlut[sc2 & 0xFF]);
                const Lut t1 = lut_from_uint4(dlut[(sc2 >> 8) & 0xFF]);
                uint32_t e0[8], e1[8];
                expand8(codes.x, t0, e0);
                expand8(codes.y, t0, e0 + 4);
                expand8(codes.z, t1, e1);
                expand8(codes.w, t1, e1 + 4);
                const int row0 = atom * kAtomRows + r, row1 = row0 + 8;
                *reinterpret_cast<uint4*>(dst + sw128_offset(row0, 2 * q)) = make_uint4(e0[0], e0[1], e0[2], e0[3]);
                *reinterpret_cast<uint4*>(dst + sw128_offset(row0, 2 * q + 1)) = make_uint4(e0[4], e0[5], e0[6], e0[7]);
                *reinterpret_cast<uint4*>(dst + sw128_offset(row1, 2 * q)) = make_uint4(e1[0], e1[1], e1[2], e1[3]);
                *reinterpret_cast<uint4*>(dst + sw128_offset(row1, 2 * q + 1)) = make_uint4(e1[4], e1[5], e1[6], e1[7]);
            }
            fence_proxy_async();       // B writes visible to the MMA; raw reads before the next copy
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&deq_full[s2]);
                mbar_arrive(&tma_empty[s1]);
            }
        }
        // epilogue: lane quarter from the hardware warp index, column half from dw
        if (*hdr_flag != 0 && mbar_wait(acc_full, 0, p.status)) {
            tc_fence_after_sync();
            const int quarter = warp & 3, half = dw >> 2;
            const int64_t mrow = m0 + quarter * 32 + lane;
            #pragma unroll 1
            for (int mi = 0; mi < SUBM; ++mi) {
                const int64_t m = mrow + mi * 128;
                const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16) + mi * kBN;
                // Rows leave through store_rows32 (a 32 x 33-word tile per warp
                // in the activation ring, idle once every MMA has completed).
                uint32_t* tile = reinterpret_cast<uint32_t*>(a_ring) + (size_t)dw * (32 * 33);
                if constexpr (MODE == TcMode::kDense) {
                    // whole-row stores need 16-byte aligned rows: N % 8 == 0 and Y aligned
                    const bool vec_ok = (p.N % 8) == 0 && (reinterpret_cast<uintptr_t>(p.Y) & 15) == 0;
                    if (p.partial != nullptr) {
                        // split-K: FP32 partial rows, summed in split order afterwards
                        float* prow = p.partial + ((int64_t)blockIdx.z * p.M + m) * p.N;
                        #pragma unroll 1
                        for (int c32 = 0; c32 < 4; ++c32) {
                            const int col = half * 128 + c32 * 32;
                            const int64_t n = n0 + col;
                            uint32_t v[16], u[16];
                            tmem_ld_32x32b_x16(trow + col, v);
                            tmem_ld_32x32b_x16(trow + col + 16, u);
                            tmem_ld_wait();
                            if (n >= p.N) continue;
                            if ((p.N % 8) == 0) {
                                uint32_t w[32];
                                #pragma unroll
                                for (int i = 0; i < 16; ++i) { w[i] = v[i]; w[16 + i] = u[i]; }
                                store_rows32(tile, w, m < m_end ? reinterpret_cast<uint32_t*>(prow + n) : nullptr,
                                             (int)(p.N - n < 32 ? p.N - n : 32), lane);
                            } else if (m < m_end) {
                                #pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (n + i < p.N) prow[n + i] = __uint_as_float(i < 16 ? v[i] : u[i - 16]);
                            }
                        }
                    } else {
                        uint16_t* yrow = p.Y + m * p.N;
                        #pragma unroll 1
                        for (int c64 = 0; c64 < 2; ++c64) {
                            const int col = half * 128 + c64 * 64;
                            const int64_t n = n0 + col;
                            uint32_t w[32];
                            #pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t v[16];
                                tmem_ld_32x32b_x16(trow + col + 16 * q, v);
                                tmem_ld_wait();
                                #pragma unroll
                                for (int i = 0; i < 8; ++i) w[8 * q + i] = pack_act2(v[2 * i], v[2 * i + 1], F16);
                            }
                            if (n >= p.N) continue;
                            if (vec_ok) {
                                store_rows32(tile, w, m < m_end ? reinterpret_cast<uint32_t*>(yrow + n) : nullptr,
                                             (int)((p.N - n) / 2 < 32 ? (p.N - n) / 2 : 32), lane);
                            } else if (m < m_end) {
                                #pragma unroll
                                for (int i = 0; i < 64; ++i)
                                    if (n + i < p.N) yrow[n + i] = (uint16_t)(w[i >> 1] >> ((i & 1) * 16));
                            }
                        }
                    }
                } else if constexpr (MODE == TcMode::kMoeFc1) {
                    // columns [0,128) are gate, [128,256) up; this warp does 64 of the 128
                    // (per-lane 32-byte stores: staging these 128-byte row pieces
                    // through shared memory measured slower)
                    #pragma unroll 1
                    for (int c16 = 0; c16 < 4; ++c16) {
                        const int col = half * 64 + c16 * 16;
                        uint32_t g[16], u[16];
                        tmem_ld_32x32b_x16(trow + col, g);
                        tmem_ld_32x32b_x16(trow + 128 + col, u);
                        tmem_ld_wait();
                        if (m >= m_end) continue;
                        uint32_t packed[8];
                        #pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float h0 = silu_tc(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
                            const float h1 = silu_tc(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
                            packed[i] = pack_act2(__float_as_uint(h0), __float_as_uint(h1), F16);
                        }
                        uint16_t* hrow = p.Y + m * p.I + n0 + col;      // I and n0 are multiples of 64
                        *reinterpret_cast<uint4*>(hrow) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        *reinterpret_cast<uint4*>(hrow + 8) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    }
                } else if constexpr (MODE == TcMode::kMoeFc1Plain) {
                    // h = RN(act(v)) for 128 of the tile's 256 columns (N = I, a multiple of 64)
                    #pragma unroll 1
                    for (int c64 = 0; c64 < 2; ++c64) {
                        const int col = half * 128 + c64 * 64;
                        const int64_t n = n0 + col;
                        uint32_t w[32];
                        #pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t v[16];
                            tmem_ld_32x32b_x16(trow + col + 16 * q, v);
                            tmem_ld_wait();
                            #pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float h0 = plain_act_tc(__uint_as_float(v[2 * i]), p.act);
                                const float h1 = plain_act_tc(__uint_as_float(v[2 * i + 1]), p.act);
                                w[8 * q + i] = pack_act2(__float_as_uint(h0), __float_as_uint(h1), F16);
                            }
                        }
                        if (n >= p.N) continue;
                        store_rows32(tile, w, m < m_end ? reinterpret_cast<uint32_t*>(p.Y + m * p.N + n) : nullptr, 32,
                                     lane);
                    }
                } else {
                    // p * y rows per routing slot, through the shared-memory tile as
                    // store_rows32 does, with the row's slot shuffled instead of a
                    // pointer (N a multiple of 16)
                    const int32_t slot = m < m_end ? p.perm[m] : -1;
                    const float wt = m < m_end ? p.wts[slot] : 0.0f;
                    float* ftile = reinterpret_cast<float*>(tile);
                    #pragma unroll 1
                    for (int c32 = 0; c32 < 4; ++c32) {
                        const int col = half * 128 + c32 * 32;
                        uint32_t v[16], u[16];
                        tmem_ld_32x32b_x16(trow + col, v);
                        tmem_ld_32x32b_x16(trow + col + 16, u);
                        tmem_ld_wait();
                        #pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            ftile[lane * 33 + i] = wt * __uint_as_float(v[i]);
                            ftile[lane * 33 + 16 + i] = wt * __uint_as_float(u[i]);
                        }
                        __syncwarp();
                        const int64_t n = n0 + col + (lane & 7) * 4;
                        #pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int r = i * 4 + (lane >> 3);
                            const int32_t sl = __shfl_sync(0xffffffffu, slot, r);
                            const float* src = ftile + r * 33 + (lane & 7) * 4;
                            if (sl >= 0 && n < p.N)
                                *reinterpret_cast<float4*>(p.Yp + (int64_t)sl * p.N + n) =
                                    make_float4(src[0], src[1], src[2], src[3]);
                        }
                        __syncwarp();
                    }
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 256 * SUBM);
    }
}

// ------------------------------------------------------------------------
// Dense tile GEMM with the weights as the tensor-memory A operand.
//
// The kernel above writes the dequantized weights into shared memory, where
// they compete with the MMAs' own operand reads for shared-memory bandwidth
// (removing those stores alone made it ~20% faster on GB300).  Here the dequant
// threads write them straight into tensor memory with tcgen05.st, and the MMA
// takes A from there: D[weight row, token] = W x X^T.
//
// One CTA covers 256 weight rows x NT tokens (NT = 128 or 192) over its K range:
//   warp 0       producer: per 64-k block, a TMA tile load of the activations
//                (NT rows x 64 k, 128-byte swizzle, zero fill past M and K) and a
//                bulk copy of the raw 256-row weight block into a kWaS1-stage ring;
//   warp 1       allocates all 512 tensor-memory columns and issues, per block,
//                2 x 4 tcgen05 MMAs (M = 128 weight rows from tensor memory,
//                N = NT tokens from shared memory, K = 16);
//   warps 2..17  dequant: a thread owns one weight row (its tensor-memory lane)
//                and half of the block's k (two 16-k groups); it reads their
//                codes and scales, expands them through the magnitude table and
//                stores 16 packed columns; afterwards the epilogue (tensor memory
//                -> registers -> Y[token, row]).
// Tensor-memory columns: accumulator of weight half s at [256 s, 256 s + NT);
// the S2 A stages (64 columns each: two halves of 32 columns = 64 k) fill the
// rest, S2 / 2 after each accumulator: 2 stages with 192-token tiles, 4 with 128.
constexpr int kWaS1 = 4;                 // activation + raw-weight ring
constexpr int kWaS2Max = 4;
template <int NT> __host__ __device__ constexpr int wa_stages() { return NT == 128 ? 4 : 2; }
constexpr int kWaDeqWarps = 16;
constexpr int kWaThreads = (kWaDeqWarps + 2) * 32;

template <int NT>
struct WaSmem {
    static constexpr size_t kXBytes = (size_t)NT * 128;                     // NT rows x 64 k
    static constexpr size_t x = 0;                                           // 1024-aligned
    static constexpr size_t raw = x + (size_t)kWaS1 * kXBytes;
    static constexpr size_t lut = raw + (size_t)kWaS1 * kBRawBytes;
    static constexpr size_t bars = lut + kLutBytes;
    static constexpr size_t misc = bars + 24 * 8;
    static constexpr size_t total = misc + 64;
};

template <int NT>
__device__ __forceinline__ uint32_t wa_a_col(int st, int s) {
    constexpr int half = wa_stages<NT>() / 2;
    return (uint32_t)((st < half ? NT + 64 * st : 256 + NT + 64 * (st - half)) + 32 * s);
}

template <int NT, bool F16>
__global__ void __launch_bounds__(kWaThreads, 1)
tc_wa_kernel(const __grid_constant__ CUtensorMap tmap_x, const TcKParams p) {
    static_assert(NT == 128 || NT == 192, "token tile");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using L = WaSmem<NT>;
    uint8_t* x_ring = smem + L::x;
    uint8_t* raw_ring = smem + L::raw;
    uint4* lut = reinterpret_cast<uint4*>(smem + L::lut);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars);
    uint64_t* tma_full = bars;                      // [kWaS1]
    uint64_t* tma_empty = bars + kWaS1;             // [kWaS1]
    constexpr int kWaS2 = wa_stages<NT>();
    uint64_t* deq_full = bars + 2 * kWaS1;             // [kWaS2]
    uint64_t* deq_empty = bars + 2 * kWaS1 + kWaS2Max; // [kWaS2]
    uint64_t* acc_full = bars + 2 * kWaS1 + 2 * kWaS2Max;
    uint64_t* lut_bar = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::misc);
    volatile int* hdr_flag = reinterpret_cast<volatile int*>(smem + L::misc + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t n0 = (int64_t)blockIdx.x * kBN;
    const int64_t m0 = (int64_t)blockIdx.y * NT;
    const int kb_first = (int)blockIdx.z * p.kb_per_split;
    const int64_t kb_left = p.KB - kb_first;
    const int nkb = (int)(kb_left < p.kb_per_split ? kb_left : p.kb_per_split);

    if (tid == 0) {
        for (int s = 0; s < kWaS1; ++s) {
            mbar_init(&tma_full[s], 1);
            mbar_init(&tma_empty[s], 1 + kWaDeqWarps);   // MMA commit + every dequant warp
        }
        for (int s = 0; s < kWaS2; ++s) {
            mbar_init(&deq_full[s], kWaDeqWarps);
            mbar_init(&deq_empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(lut_bar, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t idesc = umma_idesc(128, NT, F16);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const Header* hdr = reinterpret_cast<const Header*>(p.rp);
            const bool ok_hdr = hdr->magic == kMagic && hdr->N == p.N && hdr->K == p.K;
            *hdr_flag = ok_hdr ? 1 : 0;
            if (!ok_hdr) {
                record_status(p.status, NVFP4_ERR_BAD_WEIGHT);
                mbar_arrive(lut_bar);
            } else {
                mbar_arrive_expect_tx(lut_bar, (uint32_t)kLutBytes);
                bulk_g2s(lut, p.rp + lut_offset<F16>(), (uint32_t)kLutBytes, lut_bar);
                const uint8_t* wtile = p.rp + kTilesOffset + atom_offset(n0 / kTileRows, 0, 0, p.KB);
                int issued = 0;
                for (int kb = 0; kb < nkb; ++kb) {
                    const int s = kb % kWaS1;
                    if (kb >= kWaS1 && !mbar_wait(&tma_empty[s], ((kb / kWaS1) - 1) & 1, p.status)) break;
                    mbar_arrive_expect_tx(&tma_full[s], (uint32_t)L::kXBytes + kBRawBytes);
                    tma_load_2d(x_ring + (size_t)s * L::kXBytes, &tmap_x, (kb_first + kb) * 64, (int)m0, &tma_full[s]);
                    bulk_g2s(raw_ring + (size_t)s * kBRawBytes, wtile + (size_t)(kb_first + kb) * kBRawBytes,
                             kBRawBytes, &tma_full[s]);
                    ++issued;
                }
                // no copy may still target this CTA when it exits
                mbar_wait(lut_bar, 0, p.status);
                for (int kb = issued > kWaS1 ? issued - kWaS1 : 0; kb < issued; ++kb)
                    mbar_wait(&tma_full[kb % kWaS1], (kb / kWaS1) & 1, p.status);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            bool ok = mbar_wait(lut_bar, 0, p.status) && *hdr_flag != 0;
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s1 = kb % kWaS1, s2 = kb % kWaS2;
                ok = mbar_wait(&tma_full[s1], (kb / kWaS1) & 1, p.status) &&
                     mbar_wait(&deq_full[s2], (kb / kWaS2) & 1, p.status);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t x_base = smem_u32(x_ring + (size_t)s1 * L::kXBytes);
                #pragma unroll
                for (int s = 0; s < 2; ++s)
                    #pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f16kind_ts(tmem + 256 * s, tmem + wa_a_col<NT>(s2, s) + 8 * kk,
                                        sw128_kmajor_desc(x_base + kk * 32), idesc, (kb | kk) != 0);
                umma_commit(&tma_empty[s1]);
                umma_commit(&deq_empty[s2]);
            }
            umma_commit(acc_full);          // also waits out every MMA issued above
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ dequant, then epilogue
        // Warp -> (lane quarter Q: the hardware warp index decides which 32
        // tensor-memory lanes a warp may access; weight half s; group pair gp).
        // Lane t = (a, h, r) -> atom 8s + 2Q + a, row r + 8h of that atom; the
        // row's group j codes are the 8 bytes at 16 (4r + j) + 8h of the atom.
        // Loading the pair in an order rotated by r spreads a half warp's
        // 8-byte loads over 8 bank pairs.
        const int idx = (warp - 2) >> 2, Q = warp & 3;
        const int s = idx >> 1, gp = idx & 1;
        const int a = lane & 1, h = (lane >> 1) & 1, r = (lane >> 2) & 7;
        const int atom = 8 * s + 2 * Q + a;
        const int n_local = 128 * s + 32 * Q + 16 * a + 8 * h + r;
        const uint32_t lane_addr = (uint32_t)(32 * Q) << 16;
        const int rot = r & 1;
        bool ok = mbar_wait(lut_bar, 0, p.status) && *hdr_flag != 0;
        for (int kb = 0; kb < nkb && ok; ++kb) {
            const int s1 = kb % kWaS1, s2 = kb % kWaS2;
            ok = mbar_wait(&tma_full[s1], (kb / kWaS1) & 1, p.status);
            if (ok && kb >= kWaS2) ok = mbar_wait(&deq_empty[s2], ((kb / kWaS2) - 1) & 1, p.status);
            if (!ok) break;
            tc_fence_after_sync();
            const uint8_t* at = raw_ring + (size_t)s1 * kBRawBytes + atom * kAtomBytes;
            const uint2 v0 = *reinterpret_cast<const uint2*>(at + 16 * (4 * r + 2 * gp + rot) + 8 * h);
            const uint2 v1 = *reinterpret_cast<const uint2*>(at + 16 * (4 * r + 2 * gp + (rot ^ 1)) + 8 * h);
            const uint2 g0 = rot ? v1 : v0, g1 = rot ? v0 : v1;
            // scales of groups 2gp, 2gp + 1: bytes 2 (2gp + i) + h of the 8 at 512 + 8r
            const uint32_t sc = *reinterpret_cast<const uint32_t*>(at + kAtomCodeBytes + 8 * r + 4 * gp) >> (8 * h);
            const Lut t0 = lut_from_uint4(lut[sc & 0xFFu]);
            const Lut t1 = lut_from_uint4(lut[(sc >> 16) & 0xFFu]);
            uint32_t e[16];
            expand8(g0.x, t0, e);
            expand8(g0.y, t0, e + 4);
            expand8(g1.x, t1, e + 8);
            expand8(g1.y, t1, e + 12);
            tmem_st_32x32b_x16(tmem + lane_addr + wa_a_col<NT>(s2, s) + 16 * gp, e);
            tmem_st_wait();
            tc_fence_before_sync();
            fence_proxy_async();       // raw reads before the next copy into the stage
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&deq_full[s2]);
                mbar_arrive(&tma_empty[s1]);
            }
        }
        // epilogue: this thread's row of the half-s accumulator, half gp of the NT tokens
        if (*hdr_flag != 0 && mbar_wait(acc_full, 0, p.status)) {
            tc_fence_after_sync();
            const int64_t n = n0 + n_local;
            const bool n_ok = n < p.N;
            const uint32_t trow = tmem + lane_addr + 256 * s;
            #pragma unroll 1
            for (int c16 = gp * (NT / 32); c16 < (gp + 1) * (NT / 32); ++c16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(trow + c16 * 16, v);
                tmem_ld_wait();
                const int64_t mb = m0 + c16 * 16;
                if (!n_ok || mb >= p.M) continue;
                const int cnt = p.M - mb < 16 ? (int)(p.M - mb) : 16;
                if (p.partial != nullptr) {
                    float* col = p.partial + ((int64_t)blockIdx.z * p.M + mb) * p.N + n;
                    #pragma unroll
                    for (int i = 0; i < 16; ++i, col += p.N)
                        if (i < cnt) *col = __uint_as_float(v[i]);
                } else {
                    uint16_t* col = p.Y + mb * p.N + n;
                    #pragma unroll
                    for (int i = 0; i < 16; ++i, col += p.N)
                        if (i < cnt) *col = f32_to_act_bits<F16>(__uint_as_float(v[i]));
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

// Y = RN(sum over splits of the FP32 partials) in the activation type, splits in order.
template <bool F16>
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, int64_t MN,
                                     uint16_t* __restrict__ Y) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= MN) return;
    float4 s = *reinterpret_cast<const float4*>(part + i);
    for (int k = 1; k < splits; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(part + (int64_t)k * MN + i);
        s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    // Y is only guaranteed 4-byte aligned: two 32-bit stores
    reinterpret_cast<uint32_t*>(Y + i)[0] = (uint32_t)f32_to_act_bits<F16>(s.x) | ((uint32_t)f32_to_act_bits<F16>(s.y) << 16);
    reinterpret_cast<uint32_t*>(Y + i)[1] = (uint32_t)f32_to_act_bits<F16>(s.z) | ((uint32_t)f32_to_act_bits<F16>(s.w) << 16);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

nvfp4_status encode_rows_map(CUtensorMap* tmap, const uint16_t* X, int64_t rows, int64_t K, bool f16,
                             uint32_t box_rows = 128) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(NVFP4_ERR_CUDA, "tile GEMM: cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult cr = enc(tmap, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(X), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "tile GEMM: tensor map encode failed (%d)", (int)cr);
    return NVFP4_OK;
}

template <int SUBM, TcMode MODE, bool F16>
nvfp4_status launch_tc_typed(const uint16_t* X, int64_t x_rows, const TcKParams& kp, dim3 grid, cudaStream_t stream) {
    CUtensorMap tmap;
    nvfp4_status st = encode_rows_map(&tmap, X, x_rows, kp.K, F16);
    if (st != NVFP4_OK) return st;
    const size_t smem = TcSmem<SUBM>::total + 1024;
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<SUBM, MODE, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return check_cuda(e, "tile GEMM: shared memory attribute");
    tc_gemm_kernel<SUBM, MODE, F16><<<grid, kTcThreads, smem, stream>>>(tmap, kp);
    return check_cuda(cudaGetLastError(), "tile GEMM: launch");
}

template <int SUBM, TcMode MODE>
nvfp4_status launch_tc_impl(const uint16_t* X, int64_t x_rows, const TcKParams& kp, dim3 grid, bool f16,
                            cudaStream_t stream) {
    return f16 ? launch_tc_typed<SUBM, MODE, true>(X, x_rows, kp, grid, stream)
               : launch_tc_typed<SUBM, MODE, false>(X, x_rows, kp, grid, stream);
}

template <int NT, bool F16>
nvfp4_status launch_wa_typed(const uint16_t* X, const TcKParams& kp, dim3 grid, cudaStream_t stream) {
    CUtensorMap tmap;
    nvfp4_status st = encode_rows_map(&tmap, X, kp.M, kp.K, F16, NT);
    if (st != NVFP4_OK) return st;
    // The kernel takes all 512 tensor-memory columns: request enough shared
    // memory that a second CTA, which would have to wait for them, never
    // becomes resident on the same SM.
    constexpr size_t kOneCtaPerSm = 116 * 1024;
    const size_t smem = WaSmem<NT>::total + 1024 > kOneCtaPerSm ? WaSmem<NT>::total + 1024 : kOneCtaPerSm;
    cudaError_t e = cudaFuncSetAttribute(tc_wa_kernel<NT, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return check_cuda(e, "tile GEMM: shared memory attribute");
    tc_wa_kernel<NT, F16><<<grid, kWaThreads, smem, stream>>>(tmap, kp);
    return check_cuda(cudaGetLastError(), "tile GEMM: launch");
}

template <int NT>
nvfp4_status launch_wa(const uint16_t* X, const TcKParams& kp, dim3 grid, bool f16, cudaStream_t stream) {
    return f16 ? launch_wa_typed<NT, true>(X, kp, grid, stream) : launch_wa_typed<NT, false>(X, kp, grid, stream);
}

size_t awq_ws_bytes(int64_t M, int64_t K) { return (size_t)round_up(M * K * 2, 256); }

// Plan of a dense tile GEMM: which of the two tile kernels, its token tile
// and its split of K, from a cost model fitted to GB300 timings.  A wave of
// CTAs costs t_blk per 64-k block plus 3 us: 0.82 us for the shared-memory
// kernel's 256-token tiles (0.74 us for 128), 0.64 us for the tensor-memory-A
// kernel's tiles of 192 or 128 tokens -- about the same cost per FLOP, so the
// choice mostly follows how evenly each tiling fills the SMs.  A K split adds
// its FP32 partials' write and read at ~6 TB/s plus a 2 us reduction; K is
// split (<= 8 ways, >= 12 blocks per split) only when the model predicts at
// least 10% less time (M=2048, K=13824, N=5120: 220 tiles of 216 blocks fill
// 1.45 waves; a 2-way split measured 235 us against 272 us).
struct TcPlan {
    bool wa;        // tensor-memory-A kernel (else shared-memory operands)
    int tok;        // tokens per tile: 128 / 256 (SUBM 1 / 2) or 128 / 192 (NT)
    int splits, kbs;
};

TcPlan plan_tc(int64_t M, int64_t N, int64_t K, double* predicted_us = nullptr) {
    const int64_t KB = round_up(K, kBlockK) / kBlockK;
    const int64_t sms = sm_count();
    auto split_plan = [&](TcPlan pl, double t_blk, double* cost_out) {
        const int64_t tiles = ceil_div(N, kBN) * ceil_div(M, pl.tok);
        auto cost = [&](int64_t sp) {
            const int64_t kbs = ceil_div(KB, sp);
            double t = (double)ceil_div(tiles * sp, sms) * ((double)kbs * t_blk + 3.0);
            if (sp > 1) t += 2.0 * (double)sp * (double)M * (double)N * 4.0 / 6.0e6 + 2.0;
            return t;
        };
        pl.splits = 1;
        pl.kbs = (int)KB;
        double best_t = cost(1);
        if ((M % 4) == 0 && (N % 4) == 0) {
            const double limit = 0.9 * best_t;
            for (int sp = 2; sp <= 8 && KB / sp >= 12; ++sp) {
                const double t = cost(sp);
                if (t < limit && t < best_t) { best_t = t; pl.splits = sp; pl.kbs = (int)ceil_div(KB, sp); }
            }
            if (pl.splits > 1) pl.splits = (int)ceil_div(KB, pl.kbs);
        }
        *cost_out = best_t;
        return pl;
    };
    double t_sm, t_wa;
    const int sub = M <= 128 ? 1 : 2;
    const TcPlan sm = split_plan(TcPlan{false, 128 * sub, 1, 1}, sub == 1 ? 0.74 : 0.82, &t_sm);
    const int nt = ceil_div(M, 192) < ceil_div(M, 128) ? 192 : 128;
    const TcPlan wa = split_plan(TcPlan{true, nt, 1, 1}, 0.64, &t_wa);
    if (predicted_us) *predicted_us = t_wa < t_sm ? t_wa : t_sm;
    return t_wa < t_sm ? wa : sm;
}

}  // namespace

void tc_plan_info(int64_t M, int64_t N, int64_t K, bool* wa, int* tokens, int* splits) {
    const TcPlan pl = plan_tc(M, N, K);
    *wa = pl.wa;
    *tokens = pl.tok;
    *splits = pl.splits;
}

// Streaming kernel or tile kernels for M > 16: whichever a cost model predicts
// faster.  The streaming kernel expands every weight once per 16 tokens (its
// token chunks run as separate CTAs): about 4 us plus one 16-token pass over
// the weights at 4.8 T weights/s on GB300 (M = 32..300, N = 1000..14336,
// K = 720..14336, within 15 %); the tile kernels' time is their plan's
// (wave-quantized blocks plus the K split's reduction pass).  From M = 512 the
// tiles always win.
bool tc_tiles_fill(int64_t M, int64_t N) {
    if (M <= 16) return false;
    const int64_t tiles = ceil_div(N, kBN) * (M <= 128 ? ceil_div(M, 128) : ceil_div(M, 256));
    return tiles >= sm_count() / 2 || M >= 512;
}

bool use_tc_path(int64_t M, int64_t N, int64_t K) {
    if (M <= 16) return false;
    if (M >= 512) return true;
    double t_tile = 0.0;
    plan_tc(M, N, K, &t_tile);
    const double t_stream = 4.0 + (double)ceil_div(M, 16) * (double)N * (double)K / 4.8e6;
    return t_tile < t_stream;
}

size_t tc_workspace_bytes(int64_t M, int64_t N, int64_t K, bool has_pqs) {
    const TcPlan sp = plan_tc(M, N, K);
    const size_t part = sp.splits > 1 ? (size_t)round_up((int64_t)sp.splits * M * N * 4, 256) : 0;
    return (has_pqs ? awq_ws_bytes(M, K) : 0) + part;
}

nvfp4_status launch_tc(const TcParams& p, cudaStream_t stream) {
    const uint16_t* X = p.X;
    if (p.pqs) {
        nvfp4_status st = launch_awq_scale(p.X, p.pqs, (uint16_t*)p.workspace, p.M, p.K, p.f16, stream);
        if (st != NVFP4_OK) return st;
        X = (const uint16_t*)p.workspace;
    }
    TcKParams kp{};
    kp.rp = p.rp; kp.Y = p.Y; kp.M = p.M; kp.N = p.N; kp.K = p.K;
    kp.KB = round_up(p.K, kBlockK) / kBlockK;
    kp.status = p.status;
    const TcPlan sp = plan_tc(p.M, p.N, p.K);
    kp.kb_per_split = sp.kbs;
    if (sp.splits > 1)
        kp.partial = reinterpret_cast<float*>((uint8_t*)p.workspace + (p.pqs ? awq_ws_bytes(p.M, p.K) : 0));
    const dim3 grid((unsigned)ceil_div(p.N, kBN), (unsigned)ceil_div(p.M, sp.tok), sp.splits);
    nvfp4_status st;
    if (sp.wa)
        st = sp.tok == 192 ? launch_wa<192>(X, kp, grid, p.f16, stream) : launch_wa<128>(X, kp, grid, p.f16, stream);
    else if (sp.tok == 128)
        st = launch_tc_impl<1, TcMode::kDense>(X, p.M, kp, grid, p.f16, stream);
    else
        st = launch_tc_impl<2, TcMode::kDense>(X, p.M, kp, grid, p.f16, stream);
    if (st != NVFP4_OK || sp.splits == 1) return st;
    const int64_t MN = p.M * p.N;
    const unsigned rgrid = (unsigned)ceil_div(MN / 4, 256);
    if (p.f16) splitk_reduce_kernel<true><<<rgrid, 256, 0, stream>>>(kp.partial, sp.splits, MN, p.Y);
    else splitk_reduce_kernel<false><<<rgrid, 256, 0, stream>>>(kp.partial, sp.splits, MN, p.Y);
    return check_cuda(cudaGetLastError(), "tile GEMM: split-K reduction launch");
}

nvfp4_status launch_tc_moe(const TcMoeParams& m, cudaStream_t stream) {
    TcKParams kp{};
    kp.rp = m.w; kp.w_stride = m.w_stride; kp.items = m.items; kp.n_items = m.n_items;
    kp.M = m.rows; kp.half_stride = m.half_stride; kp.act = m.act;
    kp.perm = m.perm; kp.wts = m.wts; kp.I = m.I; kp.status = m.status;
    kp.N = m.N; kp.K = m.K; kp.KB = round_up(m.K, kBlockK) / kBlockK;
    kp.kb_per_split = (int)kp.KB;
    const bool gated_fc1 = m.fc1 && m.act == 0, plain_fc1 = m.fc1 && m.act != 0;
    kp.Y = m.H; kp.Yp = m.Yp;
    const unsigned gx = gated_fc1 ? (unsigned)(m.I / 128) : (unsigned)ceil_div(m.N, kBN);
    const dim3 grid(gx, (unsigned)m.max_items);
    if (m.subm == 1)
        return gated_fc1 ? launch_tc_impl<1, TcMode::kMoeFc1>(m.X, m.x_rows, kp, grid, m.f16, stream)
             : plain_fc1 ? launch_tc_impl<1, TcMode::kMoeFc1Plain>(m.X, m.x_rows, kp, grid, m.f16, stream)
                         : launch_tc_impl<1, TcMode::kMoeFc2>(m.X, m.x_rows, kp, grid, m.f16, stream);
    return gated_fc1 ? launch_tc_impl<2, TcMode::kMoeFc1>(m.X, m.x_rows, kp, grid, m.f16, stream)
         : plain_fc1 ? launch_tc_impl<2, TcMode::kMoeFc1Plain>(m.X, m.x_rows, kp, grid, m.f16, stream)
                     : launch_tc_impl<2, TcMode::kMoeFc2>(m.X, m.x_rows, kp, grid, m.f16, stream);
}

}  // namespace nvfp4
