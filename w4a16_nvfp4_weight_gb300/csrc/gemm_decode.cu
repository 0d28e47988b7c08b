// Decode-shaped W4A16 GEMM (few tokens): split-K, HBM-streaming, with the
// dequant fused into the tensor-core operand registers.
//
// The weight is the only large operand, so every byte of it is read once.  A
// CTA owns 128 weight rows (8 consumer warps x 16 rows; 64 rows with 4 warps
// for grids that would otherwise fill less than a wave) and one K slice.  A
// producer warp streams the slice through a shared-memory ring with bulk
// (TMA) copies: per stage three or four 64-k blocks of weights (contiguous
// 576 bytes per 16 rows) and the matching activation chunk, one copy per token
// row.  Per 64-k atom a lane reads 16 code bytes and 2 scale bytes, looks its
// two group tables up and expands the codes straight into mma.sync A
// fragments (weights on the M side, tokens on the N side).  Within a
// 16-element group the MMA's k order is permuted so that one lane consumes one
// whole group of one row per four MMAs; the activation fragments follow the
// same permutation, so the dot products are unchanged.  K is split across the
// CTAs of a thread-block cluster, which reduce their FP32 partials through
// distributed shared memory in rank order: deterministic, and no global
// workspace.  The partials travel as asynchronous stores counted on the
// receiving CTA's barrier, so no cluster-wide barrier closes the kernel: a CTA
// leaves as soon as its own pushes are out and its own share has arrived.  The AWQ pre-quant scale, when present, is applied to each ring
// stage's activation rows in shared memory, once, by the consumer warps
// together (each loads its share of the scales a stage ahead): x' = RN(x * s)
// in BF16 (or FP16), one packed multiply per pair, no extra pass and no
// workspace.
//
// The kernel is launched with programmatic dependent launch: it lets the next
// kernel of the stream start early, and it streams its first weight stages
// before waiting for the previous kernel; activations are read only after
// that wait.
//
// Method: "[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt on Hopper"
// (Description / Changes table: dequantize the NVFP4 weight each forward step
// and run a BF16 GEMM); AWQ activation scaling from "[None][fix] Apply the
// NVFP4_AWQ pre-quant scale in MegaMoE CuteDSL" (Description).
#include <algorithm>
#include <mutex>


#include "common.cuh"
#include "gemm_decode.cuh"
#include "ptx.cuh"
#include "stream_mma.cuh"


namespace nvfp4 {

namespace {

// CTA shape: W consumer warps of 16 weight rows each (W = 8: 128 rows; W = 4:
// 64 rows, for grids that would otherwise fill less than a wave) + 1 producer.
template <int W> struct Cta {
    static constexpr int kWarps = W;
    static constexpr int kThreads = (W + 1) * 32;
    static constexpr int kRowsPerCta = W * kAtomRows;
    static constexpr uint32_t kBlockBytes = W * kAtomBytes;      // W x 576: one 64-k block, contiguous
};

// Ring shape per number of 8-token MMA tiles (MT), ring kind and CTA shape:
// stages x 64-k blocks per stage.  Larger stages amortise the per-stage
// barrier work; with 16 tokens the activation chunks are twice as large, and
// two stages keep three 128-row CTAs resident per SM.  The shallow rings fit
// more CTAs per SM.  The shapes were chosen by timing the alternatives on
// GB300 over the decode layer shapes.
template <int MT, int R, int W> struct Ring;
template <> struct Ring<1, kRingDeep, 8> { static constexpr int kStages = 3, kBlocksPerStage = 4; };
template <> struct Ring<2, kRingDeep, 8> { static constexpr int kStages = 2, kBlocksPerStage = 4; };
template <> struct Ring<1, kRingShallow, 8> { static constexpr int kStages = 2, kBlocksPerStage = 4; };
template <> struct Ring<2, kRingShallow, 8> { static constexpr int kStages = 2, kBlocksPerStage = 3; };
// 64-row CTAs: four per SM (a grid of 512 such CTAs then covers 128 SMs
// evenly instead of stacking five on fewer SMs)
template <> struct Ring<1, kRingDeep, 4> { static constexpr int kStages = 3, kBlocksPerStage = 4; };
template <> struct Ring<2, kRingDeep, 4> { static constexpr int kStages = 3, kBlocksPerStage = 3; };
template <> struct Ring<1, kRingShallow, 4> { static constexpr int kStages = 2, kBlocksPerStage = 4; };
template <> struct Ring<2, kRingShallow, 4> { static constexpr int kStages = 2, kBlocksPerStage = 3; };

template <int MT, int R, int W>
using RingGeom = StreamRing<MT, Ring<MT, R, W>::kStages, Ring<MT, R, W>::kBlocksPerStage, W>;

struct Smem {
    // offsets in bytes from the dynamic shared memory base
    static constexpr size_t bars = 0;              // full[S], empty[S], lut_bar, red_bar
    static constexpr size_t flag = 120;            // header accepted (written by the producer)
    static constexpr size_t lut = 128;
    static constexpr size_t ring = lut + kLutBytes;
};

template <int MT, int R, bool F16, int W, bool AWQ>
__global__ void __launch_bounds__(Cta<W>::kThreads)
decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    using G = RingGeom<MT, R, W>;
    constexpr int kWarps = Cta<W>::kWarps;
    constexpr int kThreads = Cta<W>::kThreads;
    constexpr int kRowsPerCta = Cta<W>::kRowsPerCta;
    constexpr uint32_t kBlockBytes = Cta<W>::kBlockBytes;
    constexpr int TOK = G::kTok;
    constexpr int kStages = G::kStages;
    constexpr int kBlocksPerStage = G::kBlocksPerStage;
    constexpr uint32_t kWeightStageBytes = G::kWeightStageBytes;
    constexpr int kXRowElems = G::kXRowElems;
    constexpr size_t kStageBytes = G::kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::bars);
    uint64_t* empty = full + kStages;
    uint64_t* lut_bar = empty + kStages;
    uint64_t* red_bar = lut_bar + 1;       // this CTA's share of the split-K partials has landed
    volatile int* hdr_flag = reinterpret_cast<volatile int*>(smem + Smem::flag);
    uint4* lut = reinterpret_cast<uint4*>(smem + Smem::lut);
    uint8_t* ring = smem + Smem::ring;
    float* part = reinterpret_cast<float*>(ring + kStages * kStageBytes);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = blockIdx.x;
    const int split = blockIdx.y;
    const int64_t m0 = (int64_t)blockIdx.z * TOK;

    const int kb0 = split * p.kbs;
    const int kb1 = min(kb0 + p.kbs, (int)p.KB);
    const int nkb = kb1 - kb0;
    const int nst = (nkb + kBlocksPerStage - 1) / kBlocksPerStage;
    const int64_t m_left = p.M - m0;
    const int rows_x = (int)(m_left < TOK ? m_left : TOK);           // token rows with data (>= 1)
    const int64_t nt = ((int64_t)rg * kRowsPerCta) / kTileRows;
    const int rb0 = (rg * kRowsPerCta) % kTileRows / kAtomRows;      // first 16-row block in the tile
    const uint8_t* wsrc = p.rp + kTilesOffset + atom_offset(nt, kb0, rb0, p.KB);
    const size_t kb_stride = (size_t)kAtomsPerTileK * kAtomBytes;

    if (tid == 0) {
        pdl_launch_dependents();          // the next GEMM may start its weight prefetch
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init(lut_bar, 1);
        mbar_init(red_bar, 1);
        fence_mbar_init();
    }
    // Zero every activation chunk once: token rows without data and the k tail
    // past K are never written by a copy, so they read as zeros (or, for the
    // k tail, as earlier values of the same row, which meet zero weights).
    for (int s = 0; s < kStages; ++s) {
        uint4* xsb = reinterpret_cast<uint4*>(ring + s * kStageBytes + kWeightStageBytes);
        for (int i = tid; i < (int)(G::kXStageBytes / 16); i += kThreads) xsb[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();      // these generic writes before later bulk copies into the same bytes
    __syncthreads();
    // The split-K partials are pushed into other CTAs' shared memory at the end:
    // their barriers must be initialised first.  Arrive now, wait just before
    // the first push (by then every CTA of the cluster has long arrived).
    cluster_arrive();

    float acc[MT][4];
    #pragma unroll
    for (int mt = 0; mt < MT; ++mt)
        #pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.0f;

    if (warp == kWarps) {
        // ---------------- producer: weights and activation chunks through the ring
        if (lane == 0) {
            // Check the header before touching the rest of the buffer; every CTA
            // sees the same header, so a mismatch skips the whole cluster.
            const Header* hdr = reinterpret_cast<const Header*>(p.rp);
            const bool hdr_ok = hdr->magic == kMagic && hdr->N == p.N && hdr->K == p.K;
            *hdr_flag = hdr_ok ? 1 : 0;
            if (!hdr_ok) {
                record_status(p.status, NVFP4_ERR_BAD_WEIGHT);
                mbar_arrive(lut_bar);              // release the consumers; nothing is copied
            } else {
                // Weights and the magnitude table do not depend on the preceding
                // kernel in the stream, activations may: the first stages' weight
                // copies go out before the programmatic-launch wait, every
                // activation copy after it.
                mbar_arrive_expect_tx(lut_bar, (uint32_t)kLutBytes);
                bulk_g2s(lut, p.rp + lut_offset<F16>(), (uint32_t)kLutBytes, lut_bar);
                auto stage_blocks = [&](int i) { return min(kBlocksPerStage, nkb - i * kBlocksPerStage); };
                auto stage_xk = [&](int i) {
                    const int64_t kx_left = p.K - (int64_t)(kb0 + i * kBlocksPerStage) * kBlockK;
                    const int full_k = stage_blocks(i) * kBlockK;
                    return (int)(kx_left < full_k ? kx_left : full_k);          // multiple of 16
                };
                auto issue_weights = [&](int i) {
                    const int s = i % kStages, nb = stage_blocks(i);
                    uint8_t* st = ring + s * kStageBytes;
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(nb * kBlockBytes + (size_t)rows_x * stage_xk(i) * 2));
                    for (int b = 0; b < nb; ++b)
                        bulk_g2s(st + b * kBlockBytes, wsrc + (size_t)(i * kBlocksPerStage + b) * kb_stride,
                                 kBlockBytes, &full[s]);
                };
                auto issue_x = [&](int i) {
                    const int s = i % kStages, xk = stage_xk(i);
                    const int64_t kx = (int64_t)(kb0 + i * kBlocksPerStage) * kBlockK;
                    uint16_t* xsb = reinterpret_cast<uint16_t*>(ring + s * kStageBytes + kWeightStageBytes);
                    for (int t = 0; t < rows_x; ++t)
                        bulk_g2s(xsb + t * kXRowElems, p.X + (m0 + t) * p.K + kx, (uint32_t)xk * 2, &full[s]);
                };
                const int first = min(nst, kStages);
                for (int i = 0; i < first; ++i) issue_weights(i);
                pdl_wait_previous();
                for (int i = 0; i < first; ++i) issue_x(i);
                int issued = first;
                bool ok = true;
                for (int i = first; i < nst && ok; ++i) {
                    const int s = i % kStages;
                    ok = mbar_wait(&empty[s], ((i / kStages) - 1) & 1, p.status);
                    if (!ok) break;
                    issue_weights(i);
                    issue_x(i);
                    ++issued;
                }
                // never leave a copy in flight into this CTA's shared memory
                mbar_wait(lut_bar, 0, p.status);
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait(&full[i % kStages], (i / kStages) & 1, p.status);
            }
        }
        __syncwarp();
        cluster_wait();                   // the producer warp pairs its cluster arrival too
    } else {
        // ---------------- consumers
        const bool rows_valid = (int64_t)rg * kRowsPerCta + warp * kAtomRows < p.N;
        const int g = lane >> 2, q = lane & 3;
        bool ok = mbar_wait(lut_bar, 0, p.status) && *hdr_flag != 0;
        // the AWQ stages synchronise the consumer warps: they must all run the loop
        if constexpr (AWQ) ok = named_bar_red_and(1, kWarps * 32, ok);
        const bool work = rows_valid;
        // This lane's bytes of stage 0; stage s is kStageBytes further on.
        const uint8_t* const a0 = ring + warp * kAtomBytes;
        const uint16_t* const x0 = reinterpret_cast<const uint16_t*>(ring + kWeightStageBytes) +
                                   g * kXRowElems + q * 16;
        int s = 0;
        uint32_t phase = 0;
        const uint32_t lut_s = smem_u32(lut);
        // AWQ: k of stage i and the k it holds (a multiple of 16)
        auto stage_kx = [&](int i) { return (int64_t)(kb0 + i * kBlocksPerStage) * kBlockK; };
        auto stage_xk = [&](int i) {
            const int64_t left = p.K - stage_kx(i);
            const int full_k = min(kBlocksPerStage, nkb - i * kBlocksPerStage) * kBlockK;
            return (int)(left < full_k ? left : full_k);
        };
        using AwqStagesT = AwqStages<F16, kXRowElems, TOK, kBlocksPerStage, kWarps * 32>;
        AwqStagesT awq;
        if constexpr (AWQ) if (ok && nst > 0) awq.prefetch(p.pqs + stage_kx(0), rows_x, stage_xk(0), tid);
        for (int i = 0; i < nst && ok; ++i) {
            const bool got = mbar_wait(&full[s], phase, p.status);
            if constexpr (!AWQ) {
                if (!got) break;
            } else {
                // x' = RN(x * pre_quant_scale) once per stage, shared by the consumer
                // warps; the next stage's scales are read while this one is scaled
                AwqStagesT nxt = awq;
                if (i + 1 < nst) nxt.prefetch(p.pqs + stage_kx(i + 1), rows_x, stage_xk(i + 1), tid);
                if (got)
                    awq.apply(reinterpret_cast<uint16_t*>(ring + s * kStageBytes + kWeightStageBytes), rows_x,
                              stage_xk(i), tid);
                awq = nxt;
                // every consumer warp has scaled its share (or all stop together)
                if (!named_bar_red_and(1, kWarps * 32, got)) break;
            }
            if (work)
                stage_mma<MT, kXRowElems, F16, kBlocksPerStage, kBlockBytes>(
                    a0 + s * kStageBytes, lane, lut_s, x0 + s * (kStageBytes / 2), nkb - i * kBlocksPerStage, acc);
            fence_proxy_async();           // reads of the stage before the next bulk copy into it
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (++s == kStages) { s = 0; phase ^= 1u; }
        }

        // Push each partial of a token row with data to the CTA that reduces it:
        // output e = token * rows + row belongs to rank e / share and lands in
        // that rank's slot for this rank, counted on that rank's red_bar.  Token
        // rows past M are never sent.  No cluster-wide barrier follows: a CTA
        // leaves once its pushes are out and its own share has arrived.
        const int c = lane & 3;
        const int total = kRowsPerCta * rows_x;
        const int share = (total + p.splits - 1) / p.splits;
        const uint32_t part_s = smem_u32(part), bar_s = smem_u32(red_bar);
        cluster_wait();
        #pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            #pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int row = warp * 16 + g + (v >= 2 ? 8 : 0);
                const int t = mt * 8 + 2 * c + (v & 1);
                if (t < rows_x) {
                    const int e = t * kRowsPerCta + row;
                    const uint32_t owner = (uint32_t)(e / share);
                    st_async_b32(map_rank(part_s + 4u * (uint32_t)(split * share + e % share), owner),
                                 __float_as_uint(acc[mt][v]), map_rank(bar_s, owner));
                }
            }
        }
    }

    // Reduce this rank's share from local shared memory, ranks in order, once
    // every rank's partials for it have landed (4 bytes each).
    const int total = kRowsPerCta * rows_x;
    const int share = (total + p.splits - 1) / p.splits;
    const int e0 = split * share, e1 = min(total, e0 + share);
    if (e1 > e0) {
        if (tid == 0) mbar_arrive_expect_tx(red_bar, (uint32_t)((e1 - e0) * p.splits * 4));
        const bool got = mbar_wait_cluster(red_bar, 0, p.status);
        if (got && *hdr_flag != 0) {
            for (int e = e0 + tid; e < e1; e += kThreads) {
                float sum = 0.0f;
                for (int r = 0; r < p.splits; ++r) sum += part[r * share + (e - e0)];
                const int t = e / kRowsPerCta, row = e % kRowsPerCta;      // consecutive e -> consecutive n
                const int64_t n = (int64_t)rg * kRowsPerCta + row;
                const int64_t m = m0 + t;
                if (n < p.N && m < p.M) p.Y[m * p.N + n] = f32_to_act_bits<F16>(sum);
            }
        }
    }
}

// x' = RN(x * pre_quant_scale) in the activation type, one thread per 8 elements.
template <bool F16>
__global__ void awq_scale_kernel(const uint16_t* __restrict__ X, const uint16_t* __restrict__ pqs,
                                 uint16_t* __restrict__ Xs, int64_t M, int64_t K) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (i >= M * K) return;
    const int64_t k = i % K;
    const uint4 v = *reinterpret_cast<const uint4*>(X + i);
    const uint4 s = *reinterpret_cast<const uint4*>(pqs + k);
    const uint32_t xv[4] = {v.x, v.y, v.z, v.w};
    const uint32_t sv[4] = {s.x, s.y, s.z, s.w};
    uint32_t o[4];
    #pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint16_t lo = awq_mul<F16>((uint16_t)(xv[e] & 0xFFFF), (uint16_t)(sv[e] & 0xFFFF));
        const uint16_t hi = awq_mul<F16>((uint16_t)(xv[e] >> 16), (uint16_t)(sv[e] >> 16));
        o[e] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *reinterpret_cast<uint4*>(Xs + i) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

nvfp4_status launch_awq_scale(const uint16_t* X, const uint16_t* pqs, uint16_t* Xs, int64_t M, int64_t K,
                              bool f16, cudaStream_t stream) {
    const int64_t n8 = M * K / 8;
    if (f16) awq_scale_kernel<true><<<(unsigned)ceil_div(n8, 256), 256, 0, stream>>>(X, pqs, Xs, M, K);
    else awq_scale_kernel<false><<<(unsigned)ceil_div(n8, 256), 256, 0, stream>>>(X, pqs, Xs, M, K);
    return check_cuda(cudaGetLastError(), "AWQ activation scaling: launch");
}

template <int MT, int R, int W>
constexpr size_t smem_bytes_of() {
    // partial slots: splits x ceil(rows * TOK / splits) floats <= rows * TOK + 15 (splits <= 16)
    return Smem::ring + RingGeom<MT, R, W>::kStages * RingGeom<MT, R, W>::kStageBytes +
           ((size_t)Cta<W>::kRowsPerCta * MT * 8 + 16) * 4;
}

template <int MT, int R>
size_t smem_bytes_w(int W) { return W == 8 ? smem_bytes_of<MT, R, 8>() : smem_bytes_of<MT, R, 4>(); }

size_t decode_smem_bytes(int MT, int ring, int W) {
    if (MT == 1) return ring == kRingDeep ? smem_bytes_w<1, kRingDeep>(W) : smem_bytes_w<1, kRingShallow>(W);
    return ring == kRingDeep ? smem_bytes_w<2, kRingDeep>(W) : smem_bytes_w<2, kRingShallow>(W);
}

int decode_ctas_per_sm(int MT, int ring, int W, bool f16, bool awq) {
    // 228 KB of shared memory per SM, 1 KB of it reserved per resident CTA;
    // 2048 threads and 64 K registers per SM (registers are allocated per warp
    // in units of 256); the kernel instance's register count is read once
    constexpr size_t kSmemPerSm = 228 * 1024, kReservedPerCta = 1024;
    const size_t per_cta = decode_smem_bytes(MT, ring, W) + kReservedPerCta;
    const int by_smem = (int)(kSmemPerSm / per_cta);
    const int by_threads = 2048 / ((W + 1) * 32);
    int n = by_smem < by_threads ? by_smem : by_threads;
    const int regs = decode_kernel_regs(MT, ring, W, f16, awq);
    if (regs > 0) {
        const int per_warp = (regs * 32 + 255) / 256 * 256;
        const int by_regs = 65536 / (per_warp * (W + 1));
        n = n < by_regs ? n : by_regs;
    }
    return n < 1 ? 1 : n;
}

// The kernel instance for the activation type and AWQ choice of `p`.
template <int MT, int R, int W>
auto decode_instance(bool f16, bool awq) {
    return f16 ? (awq ? decode_kernel<MT, R, true, W, true> : decode_kernel<MT, R, true, W, false>)
               : (awq ? decode_kernel<MT, R, false, W, true> : decode_kernel<MT, R, false, W, false>);
}

template <int MT, int R, int W>
cudaError_t launch_decode_ex(const cudaLaunchConfig_t& cfg, bool f16, const DecodeParams& p) {
    return cudaLaunchKernelEx(&cfg, decode_instance<MT, R, W>(f16, p.pqs != nullptr), p);
}

template <int MT, int R, int W>
const void* decode_fn(bool f16, bool awq) {
    return (const void*)decode_instance<MT, R, W>(f16, awq);
}

// The kernel instance for (MT, ring, W): its address and a launch of it.
template <int W>
cudaError_t launch_decode_w(const cudaLaunchConfig_t& cfg, int MT, int ring, bool f16, const DecodeParams& p,
                            const void** fn_out) {
    const bool awq = p.pqs != nullptr;
    if (MT == 1) {
        if (ring == kRingDeep) {
            if (fn_out) { *fn_out = decode_fn<1, kRingDeep, W>(f16, awq); return cudaSuccess; }
            return launch_decode_ex<1, kRingDeep, W>(cfg, f16, p);
        }
        if (fn_out) { *fn_out = decode_fn<1, kRingShallow, W>(f16, awq); return cudaSuccess; }
        return launch_decode_ex<1, kRingShallow, W>(cfg, f16, p);
    }
    if (ring == kRingDeep) {
        if (fn_out) { *fn_out = decode_fn<2, kRingDeep, W>(f16, awq); return cudaSuccess; }
        return launch_decode_ex<2, kRingDeep, W>(cfg, f16, p);
    }
    if (fn_out) { *fn_out = decode_fn<2, kRingShallow, W>(f16, awq); return cudaSuccess; }
    return launch_decode_ex<2, kRingShallow, W>(cfg, f16, p);
}

int decode_kernel_regs(int MT, int ring, int W, bool f16, bool awq) {
    // registers per thread of each kernel instance, looked up once (0 when no
    // device can be asked: the caller then counts shared memory and threads)
    static int cache[2][2][2][2][2];
    static std::once_flag once[2][2][2][2][2];
    const int a = MT == 2, b = ring == kRingShallow, c = W == 4, d = f16, e = awq;
    std::call_once(once[a][b][c][d][e], [&] {
        DecodeParams dummy{};
        dummy.pqs = awq ? reinterpret_cast<const uint16_t*>(16) : nullptr;
        const void* fn = nullptr;
        cudaLaunchConfig_t cfg = {};
        if (W == 8) launch_decode_w<8>(cfg, MT, ring, f16, dummy, &fn);
        else launch_decode_w<4>(cfg, MT, ring, f16, dummy, &fn);
        cudaFuncAttributes attr{};
        cache[a][b][c][d][e] = (fn && cudaFuncGetAttributes(&attr, fn) == cudaSuccess) ? attr.numRegs : 0;
        if (cache[a][b][c][d][e] == 0) (void)cudaGetLastError();      // no device: not an error for later calls
    });
    return cache[a][b][c][d][e];
}

nvfp4_status launch_decode(const DecodeParams& p_in, int MT, int ring, int W, bool f16, cudaStream_t stream) {
    DecodeParams p = p_in;
    if (W != 8 && W != 4) return fail(NVFP4_ERR_INVALID_ARG, "decode GEMM: unsupported CTA shape %d", W);
    const int64_t rows_per_cta = (int64_t)W * kAtomRows;
    const int64_t rgs = ceil_div(p.N, rows_per_cta);
    const int64_t mchunks = ceil_div(p.M, 8 * MT);
    const size_t smem = decode_smem_bytes(MT, ring, W);
    cudaLaunchConfig_t cfg = {};
    const void* fn = nullptr;
    if (W == 8) launch_decode_w<8>(cfg, MT, ring, f16, p, &fn);
    else launch_decode_w<4>(cfg, MT, ring, f16, p, &fn);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return check_cuda(e, "decode GEMM: shared memory attribute");
    if (p.splits > 8) {            // clusters of up to 16 CTAs are not portable: opt in
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return check_cuda(e, "decode GEMM: cluster size attribute");
    }
    cfg.gridDim = dim3((unsigned)rgs, (unsigned)p.splits, (unsigned)mchunks);
    cfg.blockDim = dim3((unsigned)((W + 1) * 32), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)p.splits;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = W == 8 ? launch_decode_w<8>(cfg, MT, ring, f16, p, nullptr) : launch_decode_w<4>(cfg, MT, ring, f16, p, nullptr);
    return check_cuda(e, "decode GEMM: launch");
}

}  // namespace nvfp4
