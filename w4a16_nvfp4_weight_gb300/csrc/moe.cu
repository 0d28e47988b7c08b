// Grouped top-k MoE layer with W4A16 NVFP4 experts.
//
//   route    -- one warp per token: top-k of the FP32 router logits (ties to
//               the lower expert index, slots in descending-logit order) and
//               p = softmax over the k selected logits.
//   permute  -- one CTA: per-expert counts, offsets (exclusive scan), the
//               stable sort of the routing slots t*k+j by expert (so by expert,
//               then token, then slot) from per-expert token bitmasks (a
//               slot's place is its expert's offset plus the set bits below
//               its token), its inverse, and a list of work items (expert,
//               first permuted row, rows <= TOK).  Up to 64 tokens one CTA
//               routes and permutes.
//   fc1      -- per work item and 64 intermediate columns: the gate rows and
//               the matching up rows of the expert's FC1 weight, streamed like
//               the dense decode kernel (bulk-copy ring; with few units, split-K
//               across a cluster and a push-based reduction; with many, one
//               persistent wave walking the units with K whole); the epilogue
//               applies h = RN(silu(g) * u) and writes H in permuted row order.
//               Non-gated experts (relu2 / silu): 128 rows of [I, H] per CTA,
//               h = RN(act(v)).  With many rows per expert the tcgen05 tile
//               kernel (gemm_tc.cu) runs FC1 and FC2 instead.
//   fc2      -- the same over FC2 with H as input; the epilogue scales by the
//               slot's routing weight and writes FP32 rows per routing slot.
//   combine  -- out[t] = RN(sum over slots j of the FP32 rows), in slot
//               order.
// RN rounds to the activation type, BF16 or FP16.
// Only experts that received tokens have work items, so only their weights are
// read.  Nothing is read back to the host: the grid is sized by an upper bound
// on the number of work items, surplus CTAs exit at once, and the whole layer
// can be captured in a CUDA graph.
//
// Method: "[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt on Hopper"
// (Changes table, MoE row: dequantize only the active experts, then a BF16
// fused MoE); SGLang PR 40022 (review: gated experts carry a fused gate/up FC1);
// "[None][fix] Apply the NVFP4_AWQ pre-quant scale in MegaMoE CuteDSL"
// (Description: FC1's activation is multiplied by the pre-quant scale before
// the GEMM; a zero-token chunk launches no kernel).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemm_decode.cuh"
#include "gemm_tc.cuh"
#include "ptx.cuh"
#include "stream_mma.cuh"

namespace nvfp4 {
namespace {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopk = 16;

// ------------------------------------------------------------------- route --
// Order-preserving 32-bit key of an FP32 logit for warp max-reductions: a
// larger logit has a larger key, -0 the key of +0 (they tie), and NaN the
// smallest key (picked after every number, as a sort that puts NaN last).
__device__ __forceinline__ uint32_t logit_key(float v) {
    if (v != v) return 0u;
    const uint32_t u = __float_as_uint(v + 0.0f);          // -0 + 0 = +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp routes token t: top-k of its E logits (ties to the lower expert
// index), softmax over the selected k.  Each round every lane offers its best
// unused expert (largest key, then lowest index) and two warp reductions pick
// the winner: the largest key, then the lowest expert index among its holders.
// Lane j ends up holding selection j, written with one coalesced store.  With
// `tok_mask` (tokens mask_t0 .. mask_t0 + 63), bit t - mask_t0 of expert e's
// 64-bit mask is set for each selected expert e.
__device__ void route_token(const float* __restrict__ logits, int64_t t, int E, int topk,
                            int32_t* __restrict__ idx, float* __restrict__ wts, int lane,
                            uint32_t* tok_mask = nullptr, int64_t mask_t0 = 0) {
    constexpr int kPer = kMaxExperts / 32;
    float l[kPer];
    uint32_t key[kPer];
    uint32_t used = 0;
    #pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = lane + 32 * i;
        l[i] = e < E ? logits[t * E + e] : 0.0f;
        key[i] = logit_key(l[i]);
        if (e >= E) used |= 1u << i;
    }
    int my_e = 0;
    float my_v = 0.0f, v0 = 0.0f;
    for (int j = 0; j < topk; ++j) {
        uint32_t bk = 0u, be = 0xffffffffu;
        float bv = 0.0f;
        #pragma unroll
        for (int i = 0; i < kPer; ++i)             // ascending e: strict > keeps the lower index
            if (!((used >> i) & 1u) && (be == 0xffffffffu || key[i] > bk)) {
                bk = key[i]; be = (uint32_t)(lane + 32 * i); bv = l[i];
            }
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        const int e = (int)__reduce_min_sync(0xffffffffu, bk == kmax ? be : 0xffffffffu);
        const float v = __shfl_sync(0xffffffffu, bv, e & 31);     // the owner offered e
        if ((e & 31) == lane) used |= 1u << (e >> 5);
        if (j == lane) { my_e = e; my_v = v; }
        if (j == 0) v0 = v;                         // the first selection is the largest
    }
    // p_j = exp(v_j - v_0) / sum_j' exp(v_j' - v_0), the sum in selection order
    const float w = expf(my_v - v0);
    float sum = 0.0f;
    for (int j = 0; j < topk; ++j) sum += __shfl_sync(0xffffffffu, w, j);
    if (lane < topk) {
        idx[t * topk + lane] = my_e;
        wts[t * topk + lane] = w / sum;
        if (tok_mask != nullptr) {
            const int tb = (int)(t - mask_t0);
            atomicOr(&tok_mask[2 * my_e + (tb >> 5)], 1u << (tb & 31));
        }
    }
}

// Every kernel of the layer is launched with programmatic dependent launch:
// it lets the next kernel be scheduled early and waits for its predecessor
// (griddepcontrol.wait) before touching global memory that one may write.
__global__ void route_kernel(const float* __restrict__ logits, int64_t T, int E, int topk,
                             int32_t* __restrict__ idx, float* __restrict__ wts) {
    pdl_wait_previous();
    pdl_launch_dependents();
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (t < T) route_token(logits, t, E, topk, idx, wts, threadIdx.x & 31);
}

// ----------------------------------------------------------------- permute --
constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

// Offsets and work items from the per-expert counts cnt[0..E) in shared
// memory, by one warp: lane l scans the experts [l * per, (l + 1) * per).
// Writes off_s[e] = offsets[e], offsets[0..E] when `offsets` is not null, the
// items (expert, first permuted row, rows <= tok) when `items` is not null, and
// their count.  With tail_rows > 0 (tile path), an expert with more than tok
// rows whose last item would hold at most tail_rows rows gets that tail as an
// item of a second list, items[tail_base..] with its count in n_items[1], for
// the streaming kernels, which do not pay a whole tile for a few rows.
__device__ void expert_tables(const int32_t* cnt, int E, int tok, int32_t* __restrict__ offsets, int32_t* off_s,
                              int4* __restrict__ items, int32_t* __restrict__ n_items, int lane,
                              int tail_rows = 0, int tail_base = 0) {
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    auto is_tail = [&](int c) { return tail_rows > 0 && c > tok && c % tok != 0 && c % tok <= tail_rows; };
    int rows = 0, its = 0, tails = 0;
    for (int e = e0; e < e1; ++e) {
        const int c = cnt[e];
        rows += c;
        if (is_tail(c)) { its += c / tok; ++tails; }
        else its += (c + tok - 1) / tok;
    }
    int rows_incl = rows, its_incl = its, tails_incl = tails;
    #pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int r = __shfl_up_sync(0xffffffffu, rows_incl, off);
        const int k = __shfl_up_sync(0xffffffffu, its_incl, off);
        const int q = __shfl_up_sync(0xffffffffu, tails_incl, off);
        if (lane >= off) { rows_incl += r; its_incl += k; tails_incl += q; }
    }
    int run = rows_incl - rows, item = its_incl - its, tail = tails_incl - tails;
    for (int e = e0; e < e1; ++e) {
        const int c = cnt[e];
        if (offsets != nullptr) offsets[e] = run;
        off_s[e] = run;
        if (items != nullptr) {
            const bool t = is_tail(c);
            const int main_rows = t ? c - c % tok : c;
            for (int r = 0; r < main_rows; r += tok) items[item++] = make_int4(e, run + r, min(tok, main_rows - r), 0);
            if (t) items[tail_base + tail++] = make_int4(e, run + main_rows, c % tok, 0);
        }
        run += c;
    }
    if (lane == 31) {
        if (offsets != nullptr) offsets[E] = rows_incl;
        if (n_items != nullptr) {
            n_items[0] = its_incl;
            if (tail_rows > 0) n_items[1] = tails_incl;
        }
    }
}

// Many tokens: one CTA.  The counts come from shared-memory atomics.  The
// stable order (by expert, then token -- a token's k slots hold distinct
// experts) comes from per-expert token bitmasks, one chunk of tokens at a
// time: for each expert the running number of its slots in earlier 32-token
// words (pre), so that token t's slot of expert e lands at offsets[e] +
// pre[e][t / 32] + (set bits of its word below t).  A thread holds up to
// kPermSlots of a chunk's slots in registers, read with independent loads (a
// single-CTA loop that waited on each load in turn spent its time in memory
// latency).
constexpr int kPermSlots = 16;

__global__ void __launch_bounds__(kPermThreads)
permute_kernel(const int32_t* __restrict__ idx, int64_t T, int topk, int E, int tok, int wc,
               int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
               int4* __restrict__ items, int32_t* __restrict__ n_items, int tail_rows, int tail_base) {
    extern __shared__ uint32_t psm[];
    // rows of ws >= wc words, ws odd: the experts of one token's slots, which
    // touch the same word column, fall on different banks
    const int ws = wc | 1;
    uint32_t* mask = psm;                                            // [E][ws]
    int32_t* pre = reinterpret_cast<int32_t*>(mask + (size_t)E * ws);  // [E][ws]
    int32_t* cnt = pre + (size_t)E * ws;                             // [E]: counts, then the running base
    int32_t* off_s = cnt + E;                                        // [E]
    const int tid = threadIdx.x;
    pdl_wait_previous();
    pdl_launch_dependents();
    const int64_t n = T * topk;
    constexpr int64_t kBatch = (int64_t)kPermSlots * kPermThreads;
    for (int e = tid; e < E; e += kPermThreads) cnt[e] = 0;
    __syncthreads();
    for (int64_t b0 = 0; b0 < n; b0 += kBatch) {
        int ev[kPermSlots];
        #pragma unroll
        for (int u = 0; u < kPermSlots; ++u) {
            const int64_t i = b0 + (int64_t)u * kPermThreads + tid;
            ev[u] = i < n ? idx[i] : -1;
        }
        #pragma unroll
        for (int u = 0; u < kPermSlots; ++u)
            if (ev[u] >= 0) atomicAdd(&cnt[ev[u]], 1);
    }
    __syncthreads();
    if (tid < 32) expert_tables(cnt, E, tok, offsets, off_s, items, n_items, tid, tail_rows, tail_base);
    __syncthreads();
    for (int e = tid; e < E; e += kPermThreads) cnt[e] = 0;
    // a chunk: at most wc words of tokens and at most kBatch slots
    const int64_t ct = min((int64_t)wc * 32, kBatch / topk);
    // (the host sizes wc so that both bounds agree for the usual top-k)
    for (int64_t t0 = 0; t0 < T; t0 += ct) {
        for (int k = tid; k < E * ws; k += kPermThreads) mask[k] = 0u;
        const int64_t i0 = t0 * topk, i1 = min(T, t0 + ct) * topk;
        int ev[kPermSlots];
        #pragma unroll
        for (int u = 0; u < kPermSlots; ++u) {
            const int64_t i = i0 + (int64_t)u * kPermThreads + tid;
            ev[u] = i < i1 ? idx[i] : -1;
        }
        __syncthreads();
        #pragma unroll
        for (int u = 0; u < kPermSlots; ++u)
            if (ev[u] >= 0) {
                const int t = (int)(i0 + (int64_t)u * kPermThreads + tid) / topk - (int)t0;   // slots < 2^31
                atomicOr(&mask[ev[u] * ws + (t >> 5)], 1u << (t & 31));
            }
        __syncthreads();
        for (int e = tid; e < E; e += kPermThreads) {
            int run = cnt[e];
            for (int w = 0; w < wc; ++w) {
                pre[e * ws + w] = run;
                run += __popc(mask[e * ws + w]);
            }
            cnt[e] = run;
        }
        __syncthreads();
        #pragma unroll
        for (int u = 0; u < kPermSlots; ++u)
            if (ev[u] >= 0) {
                const int64_t i = i0 + (int64_t)u * kPermThreads + tid;
                const int t = (int)i / topk - (int)t0, e = ev[u];
                const int pos = off_s[e] + pre[e * ws + (t >> 5)] +
                                __popc(mask[e * ws + (t >> 5)] & ((1u << (t & 31)) - 1u));
                perm[pos] = (int32_t)i;
                inv[i] = pos;
            }
        __syncthreads();
    }
}

// Few tokens (T <= 64): one CTA routes every token (a warp per token) and
// builds the tables from per-expert token masks instead of counting passes:
// expert e's routed slots, in token order, are its mask's set bits, so its count
// is the mask's population and the stable position of token t's slot is
// offsets[e] + (set bits below t).  Routing, the tables and the permutation are
// three phases between two block barriers.
constexpr int64_t kFusedRouteMaxT = 64;

__global__ void __launch_bounds__(kPermThreads)
route_permute_kernel(const float* __restrict__ logits, int64_t T, int E, int topk, int tok,
                     int32_t* __restrict__ idx, float* __restrict__ wts,
                     int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                     int4* __restrict__ items, int32_t* __restrict__ n_items, int tail_rows, int tail_base) {
    __shared__ uint32_t tok_mask[2 * kMaxExperts];      // bit t: token t chose the expert
    __shared__ int32_t cnt_s[kMaxExperts];
    __shared__ int32_t off_s[kMaxExperts];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    pdl_wait_previous();
    pdl_launch_dependents();
    for (int i = tid; i < 2 * E; i += kPermThreads) tok_mask[i] = 0u;
    __syncthreads();
    for (int64_t t = w; t < T; t += kPermWarps) route_token(logits, t, E, topk, idx, wts, lane, tok_mask);
    __syncthreads();
    if (w == 0) {
        for (int e = lane; e < E; e += 32) cnt_s[e] = __popc(tok_mask[2 * e]) + __popc(tok_mask[2 * e + 1]);
        __syncwarp();
        expert_tables(cnt_s, E, tok, offsets, off_s, items, n_items, lane, tail_rows, tail_base);
    }
    __syncthreads();
    // slot i = t * topk + j of expert e: after the earlier tokens of e
    const int n = (int)T * topk;
    for (int i = tid; i < n; i += kPermThreads) {
        const int t = i / topk;
        const int e = idx[i];                // written by this CTA before the barrier
        const uint32_t lo = tok_mask[2 * e], hi = tok_mask[2 * e + 1];
        const int below = t < 32 ? __popc(lo & ((1u << t) - 1u)) : __popc(lo) + __popc(hi & ((1u << (t - 32)) - 1u));
        const int pos = off_s[e] + below;
        perm[pos] = i;
        inv[i] = pos;
    }
}

// Many tokens with a workspace: the permutation in chunks of 8 tokens, in three
// short kernels that each spread over many SMs (the single-CTA permutation
// grows by ~7.5 us per 1000 tokens: 37 us at 4096 tokens, against ~19 us for
// the three kernels, route included).  route_count_kernel routes a chunk's tokens
// (a warp per token, as route_kernel) and counts each expert's slots in it
// from per-expert token masks; chunk_scan_kernel turns each expert's counts
// over the chunks into exclusive prefixes and a total (a warp per expert);
// chunk_permute_kernel gives chunk c's slots of expert e the positions after
// the earlier chunks' slots of e, in token order -- the same stable order as
// the single-CTA kernel.
constexpr int kChunkTokens = 8;
// From this many tokens: below, the routing kernel and the single-CTA
// permutation (two launches) measured as fast as the three chunked ones.
constexpr int64_t kChunkedRouteMinT = 513;
constexpr int kChunkThreads = kChunkTokens * 32;      // a warp per token
constexpr int kScanWarps = 8;

__global__ void __launch_bounds__(kChunkThreads)
route_count_kernel(const float* __restrict__ logits, int64_t T, int E, int topk, int32_t* __restrict__ idx,
                   float* __restrict__ wts, int32_t* __restrict__ counts, int C) {
    __shared__ uint32_t tok_mask[2 * kMaxExperts];      // bit t: token t0 + t chose the expert
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int c = blockIdx.x;
    const int64_t t0 = (int64_t)c * kChunkTokens;
    pdl_wait_previous();
    pdl_launch_dependents();
    for (int i = tid; i < 2 * E; i += kChunkThreads) tok_mask[i] = 0u;
    __syncthreads();
    if (t0 + w < T) route_token(logits, t0 + w, E, topk, idx, wts, lane, tok_mask, t0);
    __syncthreads();
    // expert-major, so that one warp scans an expert's counts over the chunks coalesced
    for (int e = tid; e < E; e += kChunkThreads) counts[(int64_t)e * C + c] = __popc(tok_mask[2 * e]);
}

__global__ void __launch_bounds__(kScanWarps * 32)
chunk_scan_kernel(int32_t* __restrict__ counts, int C, int E, int32_t* __restrict__ totals) {
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
    pdl_wait_previous();
    pdl_launch_dependents();
    if (e >= E) return;
    int32_t* row = counts + (int64_t)e * C;
    int run = 0;
    for (int c0 = 0; c0 < C; c0 += 32) {
        const int v = c0 + lane < C ? row[c0 + lane] : 0;
        int incl = v;
        #pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += u;
        }
        if (c0 + lane < C) row[c0 + lane] = run + incl - v;      // earlier chunks' slots of e
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) totals[e] = run;
}

__global__ void __launch_bounds__(kChunkTokens * kMaxTopk)
chunk_permute_kernel(const int32_t* __restrict__ idx, int64_t T, int topk, int E, int tok,
                     const int32_t* __restrict__ base, const int32_t* __restrict__ totals, int C,
                     int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                     int4* __restrict__ items, int32_t* __restrict__ n_items, int tail_rows, int tail_base) {
    constexpr int kThreads = kChunkTokens * kMaxTopk;
    __shared__ uint32_t tok_mask[kMaxExperts];
    __shared__ int32_t tot_s[kMaxExperts];
    __shared__ int32_t base_s[kMaxExperts];
    __shared__ int32_t off_s[kMaxExperts];
    const int tid = threadIdx.x;
    const int c = blockIdx.x;
    const int64_t t0 = (int64_t)c * kChunkTokens;
    const int nslots = (int)(min(T - t0, (int64_t)kChunkTokens) * topk);
    pdl_wait_previous();
    pdl_launch_dependents();
    for (int e = tid; e < E; e += kThreads) {
        tok_mask[e] = 0u;
        tot_s[e] = totals[e];
        base_s[e] = base[(int64_t)e * C + c];
    }
    const int e_mine = tid < nslots ? idx[t0 * topk + tid] : -1;
    __syncthreads();
    const int t = tid / topk;                            // token of this thread's slot, within the chunk
    if (e_mine >= 0) atomicOr(&tok_mask[e_mine], 1u << t);
    if (tid < 32)
        expert_tables(tot_s, E, tok, c == 0 ? offsets : nullptr, off_s, c == 0 ? items : nullptr,
                      c == 0 ? n_items : nullptr, tid, tail_rows, tail_base);
    __syncthreads();
    if (e_mine >= 0) {
        const int pos = off_s[e_mine] + base_s[e_mine] + __popc(tok_mask[e_mine] & ((1u << t) - 1u));
        const int64_t i = t0 * topk + tid;
        perm[pos] = (int32_t)i;
        inv[i] = pos;
    }
}

// Chunks of the chunked permutation.
int64_t route_chunks(int64_t T) { return ceil_div(T, (int64_t)kChunkTokens); }

// Token words per permutation chunk: a chunk holds at most kPermSlots slots
// per thread, and its masks and prefixes take about E * wc * 8 bytes of at
// most 160 KB of shared memory.
int permute_words(int64_t T, int E, int topk) {
    const int64_t cap = std::max<int64_t>(1, (160 * 1024) / (8LL * E));
    const int64_t by_slots = std::max<int64_t>(1, (int64_t)kPermSlots * kPermThreads / topk / 32);
    return (int)std::min<int64_t>(std::min<int64_t>(ceil_div(T, 32), cap), by_slots);
}
size_t permute_smem_bytes(int E, int wc) { return ((size_t)2 * E * (wc | 1) + 2 * E) * sizeof(int); }

// ------------------------------------------------- grouped streaming linear --
constexpr int kWarps = 8;                      // 8 x 16 = 128 weight rows per CTA
constexpr int kThreads = (kWarps + 1) * 32;    // + 1 producer warp
constexpr uint32_t kBlockBytes = kStreamBlockBytes;            // 4608 per 64-k block

// Ring per number of 8-row MMA tiles, as for the dense decode kernel.
template <int MT> struct MoeRing;
template <> struct MoeRing<1> { using G = StreamRing<1, 3, 4>; };
template <> struct MoeRing<2> { using G = StreamRing<2, 2, 4>; };
template <> struct MoeRing<4> { using G = StreamRing<4, 2, 4>; };
constexpr size_t kRingOffset = 128;

struct MoeLinParams {
    const uint8_t* w;          // E repacked weights, expert e at w + e * w_stride
    size_t w_stride;
    int64_t N, K, KB;          // weight rows / inner dimension / 64-k blocks
    int kbs, splits;
    const uint16_t* X;         // gated: token activations [T, K]; else: H rows [T*k, K]
    const int32_t* perm;       // [T*k]
    int topk;
    const int4* items;         // (expert, first permuted row, rows, -); null: one dense
    const int32_t* n_items;    //   weight and consecutive runs of TOK token rows
    int64_t rows;              // dense use: token rows
    int64_t I;                 // gated: intermediate size (gate rows [0, I), up rows [I, 2I))
    size_t half_stride;        // gated: 0 = one [2I, K] weight; else bytes from the gate
                               //   shard [I, K] to the up shard [I, K] (own globals)
    int act;                   // ungated: 0 = FC2 (x p -> Yp); 1 relu2 / 2 silu FC1 -> H
    uint16_t* H;               // gated (and non-gated FC1) output [T*k, I]
    float* Yp;                 // FC2 output [T*k, N], scaled by the routing weight
    const float* wts;          // [T*k] routing weights
    const uint16_t* pqs;       // FC1: AWQ pre-quant scale [K] applied to the activation
                               //   fragments (x' = RN(x * s)); null = none
    int early;                 // 1: the routing tables were written two launches back, so
                               //   they and the weights may be read before the wait
    // single token (ONE kernels): every CTA routes the token from its logits
    const float* logits;       // [E] FP32
    int E;
    uint16_t* out;             // FC2 + combine: the layer output [N]
    int32_t* r_idx;            // FC1: the routing tables, written by CTA (0, 0, 0) when
    float* r_wts;              //   not null -- top-k experts and weights [topk], the
    int32_t* r_perm;           //   permutation and its inverse [topk], the expert
    int32_t* r_inv;            //   offsets [E + 1]
    int32_t* r_offsets;
    int* status;
};

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }

// Activation of a non-gated expert: 1 = squared ReLU, 2 = SiLU.
__device__ __forceinline__ float plain_act(float v, int act) {
    if (act == 1) {
        const float r = fmaxf(v, 0.0f);
        return r * r;
    }
    return silu_f(v);
}

// ONE = 1: FC1 of a single token, ONE = 2: its FC2 with the combine.  The
// token's routing is computed by every CTA from the logits (the same top-k
// everywhere), so no routing kernel runs: grid z is the routing slot j, whose
// expert is the j-th selection.  FC1 writes h_j to row j of H.  FC2 clusters
// the topk slots of a row group, each slot's K split over `splits` CTAs: the
// push reduction then sums p_j * y_j over the slots in slot order (each
// slot's splits in order) and writes the output row, so no combine kernel
// runs either.
template <int MT, bool GATED, bool F16, bool AWQ, int ONE = 0>
__global__ void __launch_bounds__(kThreads)
moe_linear_kernel(const MoeLinParams p) {
    __shared__ int32_t one_e[kMaxTopk];        // single token: its experts and weights
    __shared__ float one_p[kMaxTopk];
    extern __shared__ __align__(128) uint8_t smem[];
    using G = typename MoeRing<MT>::G;
    constexpr int TOK = G::kTok;
    constexpr int kStages = G::kStages;
    constexpr int kBlocksPerStage = G::kBlocksPerStage;
    constexpr uint32_t kWeightStageBytes = G::kWeightStageBytes;
    constexpr int kXRowElems = G::kXRowElems;
    constexpr size_t kStageBytes = G::kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStages;
    uint64_t* lut_bar = empty + kStages;
    uint64_t* red_bar = lut_bar + 1;          // this CTA's share of the split-K partials has landed
    volatile int* hdr_flag = reinterpret_cast<volatile int*>(smem + 120);
    // magnitude tables: one, or two with gate/up shards (gate first)
    const bool shards = GATED && p.half_stride != 0;
    uint4* lut = reinterpret_cast<uint4*>(smem + kRingOffset);
    uint8_t* ring = smem + kRingOffset + (shards ? 2 : 1) * kLutBytes;
    float* part = reinterpret_cast<float*>(ring + kStages * kStageBytes);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cgi = blockIdx.x;                // column group: 64 (gated) or 128 output features
    const int split = blockIdx.y;
    const int item_id = blockIdx.z;
    // the cluster's reduction ranks: the K splits, or (single-token FC2) the
    // slots, each with its K splits (slot-major, so the sum runs slot by slot)
    const int rank = ONE == 2 ? item_id * p.splits + split : split;
    const int nranks = ONE == 2 ? p.topk * p.splits : p.splits;
    // Items and activations come from earlier kernels.  Dependents are released
    // only after the wait: an FC2 reads the routing tables before its own wait
    // (`early`), which is safe once the kernel that wrote them, two launches
    // back, is known to be complete -- as it is when its successor has waited.
    const bool early = (p.early != 0 && p.items != nullptr) || ONE == 2;
    if (!early) {
        pdl_wait_previous();
        pdl_launch_dependents();
    }
    int4 item;                                 // the same for every CTA of the cluster
    if constexpr (ONE != 0) {
        // FC1 has waited for the logits' producer; FC2 starts only after FC1
        // has waited too, so it may route before its own wait
        if (warp == 0) route_token(p.logits, 0, p.E, p.topk, one_e, one_p, lane);
        __syncthreads();
        if (ONE == 1 && warp == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && p.r_idx != nullptr) {
            // the layer's routing outputs: slots sorted by expert (distinct)
            if (lane < p.topk) {
                int pos = 0;
                for (int j = 0; j < p.topk; ++j) pos += one_e[j] < one_e[lane];
                p.r_idx[lane] = one_e[lane];
                p.r_wts[lane] = one_p[lane];
                p.r_perm[pos] = lane;
                p.r_inv[lane] = pos;
            }
            for (int ex = lane; ex <= p.E; ex += 32) {
                int c = 0;
                for (int j = 0; j < p.topk; ++j) c += one_e[j] < ex;
                p.r_offsets[ex] = c;
            }
        }
        item = make_int4(one_e[item_id], item_id, 1, 0);
    } else if (p.items != nullptr) {
        if (item_id >= (early ? __ldcg(p.n_items) : *p.n_items)) return;
        item = early ? __ldcg(p.items + item_id) : p.items[item_id];
    } else {
        const int64_t first = (int64_t)item_id * TOK;
        if (first >= p.rows) return;
        item = make_int4(0, (int)first, (int)min((int64_t)TOK, p.rows - first), 0);
    }
    const int e = item.x, r0 = item.y, nrows = item.z;
    const uint8_t* wexp = p.w + (size_t)e * p.w_stride;

    const int kb0 = split * p.kbs;
    const int kb1 = min(kb0 + p.kbs, (int)p.KB);
    const int nkb = kb1 - kb0;
    const int nst = (nkb + kBlocksPerStage - 1) / kBlocksPerStage;
    // weight rows of this CTA: gated -> 64 gate rows + the 64 matching up rows
    // (two runs of four atoms); ungated -> 128 consecutive rows (one run of eight)
    const int64_t row_a = GATED ? (int64_t)cgi * 64 : (int64_t)cgi * 128;
    const int64_t row_b = GATED ? (shards ? 0 : p.I) + (int64_t)cgi * 64 : 0;
    const uint8_t* wup = shards ? wexp + p.half_stride : wexp;      // where the up rows live
    auto atom_src = [&](const uint8_t* base, int64_t row0, int kb) {
        const int64_t rbg = row0 / kAtomRows;
        return base + kTilesOffset + atom_offset(rbg / kAtomsPerTileK, kb, rbg % kAtomsPerTileK, p.KB);
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init(lut_bar, 1);
        mbar_init(red_bar, 1);
        fence_mbar_init();
    }
    for (int s = 0; s < kStages; ++s) {
        uint4* xsb = reinterpret_cast<uint4*>(ring + s * kStageBytes + kWeightStageBytes);
        for (int i = tid; i < TOK * kXRowElems / 8; i += kThreads) xsb[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();
    __syncthreads();
    cluster_arrive();                          // every CTA's red_bar is ready before any push

    float acc[MT][4];
    #pragma unroll
    for (int mt = 0; mt < MT; ++mt)
        #pragma unroll
        for (int v = 0; v < 4; ++v) acc[mt][v] = 0.0f;

    if (warp == kWarps) {
        if (lane == 0) {
            const Header* hdr = reinterpret_cast<const Header*>(wexp);
            const Header* hdr_up = reinterpret_cast<const Header*>(wup);
            const bool hdr_ok = hdr->magic == kMagic && hdr->N == p.N && hdr->K == p.K &&
                                (!shards || (hdr_up->magic == kMagic && hdr_up->N == p.N && hdr_up->K == p.K));
            *hdr_flag = hdr_ok ? 1 : 0;
            if (!hdr_ok) {
                record_status(p.status, NVFP4_ERR_BAD_WEIGHT);
                mbar_arrive(lut_bar);
                if (early) {
                    pdl_wait_previous();
                    pdl_launch_dependents();
                }
            } else {
                mbar_arrive_expect_tx(lut_bar, (uint32_t)((shards ? 2 : 1) * kLutBytes));
                bulk_g2s(lut, wexp + lut_offset<F16>(), (uint32_t)kLutBytes, lut_bar);
                if (shards) bulk_g2s(lut + 256, wup + lut_offset<F16>(), (uint32_t)kLutBytes, lut_bar);
                // activation row of each of this item's routed rows (FC1 reads token
                // rows through the permutation, FC2 the permuted rows of H)
                const bool token_rows = (GATED || p.act != 0) && p.perm != nullptr;
                const uint16_t* xrow[TOK];
                for (int t = 0; t < nrows; ++t) {
                    const int64_t r = r0 + t;
                    const int64_t src_row = ONE == 1 ? 0    // the single token; FC2: H row j = r
                                            : token_rows ? (int64_t)((early ? __ldcg(p.perm + r) : p.perm[r]) / p.topk) : r;
                    xrow[t] = p.X + src_row * p.K;
                }
                auto stage_xk = [&](int i) {
                    const int nb = min(kBlocksPerStage, nkb - i * kBlocksPerStage);
                    const int64_t kx_left = p.K - (int64_t)(kb0 + i * kBlocksPerStage) * kBlockK;
                    return (int)(kx_left < nb * kBlockK ? kx_left : nb * kBlockK);
                };
                auto issue_weights = [&](int i) {
                    const int s = i % kStages;
                    const int nb = min(kBlocksPerStage, nkb - i * kBlocksPerStage);
                    uint8_t* st = ring + s * kStageBytes;
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(nb * kBlockBytes + (size_t)nrows * stage_xk(i) * 2));
                    for (int b = 0; b < nb; ++b) {
                        const int kb = kb0 + i * kBlocksPerStage + b;
                        if (GATED) {
                            bulk_g2s(st + b * kBlockBytes, atom_src(wexp, row_a, kb), kBlockBytes / 2, &full[s]);
                            bulk_g2s(st + b * kBlockBytes + kBlockBytes / 2, atom_src(wup, row_b, kb), kBlockBytes / 2,
                                     &full[s]);
                        } else {
                            bulk_g2s(st + b * kBlockBytes, atom_src(wexp, row_a, kb), kBlockBytes, &full[s]);
                        }
                    }
                };
                auto issue_x = [&](int i) {
                    const int s = i % kStages, xk = stage_xk(i);
                    const int64_t kx = (int64_t)(kb0 + i * kBlocksPerStage) * kBlockK;
                    uint16_t* xsb = reinterpret_cast<uint16_t*>(ring + s * kStageBytes + kWeightStageBytes);
                    for (int t = 0; t < nrows; ++t)
                        bulk_g2s(xsb + t * kXRowElems, xrow[t] + kx, (uint32_t)xk * 2, &full[s]);
                };
                int issued = 0;
                bool ok = true;
                if (early) {
                    // the first stages' weights (and the table, above) before the
                    // wait, their activations after it
                    const int first = min(nst, kStages);
                    for (int i = 0; i < first; ++i) issue_weights(i);
                    pdl_wait_previous();
                    pdl_launch_dependents();
                    for (int i = 0; i < first; ++i) issue_x(i);
                    issued = first;
                }
                for (int i = issued; i < nst && ok; ++i) {
                    const int s = i % kStages;
                    if (i >= kStages) ok = mbar_wait(&empty[s], ((i / kStages) - 1) & 1, p.status);
                    if (!ok) break;
                    issue_weights(i);
                    issue_x(i);
                    ++issued;
                }
                mbar_wait(lut_bar, 0, p.status);
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    mbar_wait(&full[i % kStages], (i / kStages) & 1, p.status);
            }
        } else if (early) {
            pdl_wait_previous();
            pdl_launch_dependents();
        }
        __syncwarp();
        cluster_wait();
    } else {
        if (early) {
            pdl_wait_previous();
            pdl_launch_dependents();
        }
        const int g = lane >> 2, q = lane & 3;
        bool ok = mbar_wait(lut_bar, 0, p.status) && *hdr_flag != 0;
        // the AWQ stages synchronise the consumer warps: they must all run the loop
        if constexpr (AWQ) ok = named_bar_red_and(1, kWarps * 32, ok);
        const bool rows_valid = GATED || row_a + warp * kAtomRows < p.N;
        const uint4* const wlut = (shards && warp >= 4) ? lut + 256 : lut;   // warps 4-7 hold up rows
        const uint8_t* const a0 = ring + warp * kAtomBytes;
        const uint16_t* const x0 = reinterpret_cast<const uint16_t*>(ring + kWeightStageBytes) +
                                   g * kXRowElems + q * 16;
        int s = 0;
        uint32_t phase = 0;
        const uint32_t lut_s = smem_u32(wlut);
        // AWQ: k of stage i and the k it holds (a multiple of 16)
        auto stage_kx = [&](int i) { return (int64_t)(kb0 + i * kBlocksPerStage) * kBlockK; };
        auto stage_xk = [&](int i) {
            const int64_t left = p.K - stage_kx(i);
            const int full_k = min(kBlocksPerStage, nkb - i * kBlocksPerStage) * kBlockK;
            return (int)(left < full_k ? left : full_k);
        };
        using AwqStagesT = AwqStages<F16, kXRowElems, TOK, kBlocksPerStage, kWarps * 32>;
        AwqStagesT awq;
        if constexpr (AWQ) if (ok && nst > 0) awq.prefetch(p.pqs + stage_kx(0), nrows, stage_xk(0), tid);
        for (int i = 0; i < nst && ok; ++i) {
            const bool got = mbar_wait(&full[s], phase, p.status);
            if constexpr (!AWQ) {
                if (!got) break;
            } else {
                // x' = RN(x * pre_quant_scale) once per stage, shared by the consumer
                // warps; the next stage's scales are read while this one is scaled
                AwqStagesT nxt = awq;
                if (i + 1 < nst) nxt.prefetch(p.pqs + stage_kx(i + 1), nrows, stage_xk(i + 1), tid);
                if (got)
                    awq.apply(reinterpret_cast<uint16_t*>(ring + s * kStageBytes + kWeightStageBytes), nrows,
                              stage_xk(i), tid);
                awq = nxt;
                // every consumer warp has scaled its share (or all stop together)
                if (!named_bar_red_and(1, kWarps * 32, got)) break;
            }
            if (rows_valid)
                stage_mma<MT, kXRowElems, F16, kBlocksPerStage, kBlockBytes>(
                    a0 + s * kStageBytes, lane, lut_s, x0 + s * (kStageBytes / 2), nkb - i * kBlocksPerStage, acc,
                    MT == 1 ? 1 : (nrows + 7) >> 3);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (++s == kStages) { s = 0; phase ^= 1u; }
        }
        // push the partials of rows with data to the reducing CTA, as remote
        // stores counted on its red_bar (no cluster-wide barrier afterwards)
        const int c = lane & 3;
        const uint32_t part_s = smem_u32(part), bar_s = smem_u32(red_bar);
        // single-token FC2: the partials are p_j * y_j of this CTA's slot j
        const float scale = ONE == 2 ? one_p[item_id] : 1.0f;
        cluster_wait();
        if (GATED) {
            // pair (token t, column jj): gate partial from warps 0-3, up from warps 4-7
            const int total = nrows * 64;
            const int share = (total + nranks - 1) / nranks;
            #pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                #pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int row = warp * 16 + g + (v >= 2 ? 8 : 0);
                    const int t = mt * 8 + 2 * c + (v & 1);
                    const int jj = row & 63, half = row >> 6;
                    const int ei = t * 64 + jj;
                    if (t < nrows) {
                        const uint32_t owner = (uint32_t)(ei / share);
                        st_async_b32(map_rank(part_s + 4u * (uint32_t)((rank * share + ei % share) * 2 + half), owner),
                                     __float_as_uint(acc[mt][v]), map_rank(bar_s, owner));
                    }
                }
        } else {
            const int total = nrows * 128;
            const int share = (total + nranks - 1) / nranks;
            #pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                #pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int row = warp * 16 + g + (v >= 2 ? 8 : 0);
                    const int t = mt * 8 + 2 * c + (v & 1);
                    const int ei = t * 128 + row;
                    if (t < nrows) {
                        const uint32_t owner = (uint32_t)(ei / share);
                        st_async_b32(map_rank(part_s + 4u * (uint32_t)(rank * share + ei % share), owner),
                                     __float_as_uint(scale * acc[mt][v]), map_rank(bar_s, owner));
                    }
                }
        }
    }

    // this rank's share: wait for every rank's partials (4 bytes each; two
    // per output when gated), then reduce in rank order
    const int per_e = GATED ? 2 : 1;
    const int total_e = nrows * (GATED ? 64 : 128);
    const int share_e = (total_e + nranks - 1) / nranks;
    const int e0_own = rank * share_e, e1_own = min(total_e, e0_own + share_e);
    bool landed = true;
    if (e1_own > e0_own) {
        if (tid == 0) mbar_arrive_expect_tx(red_bar, (uint32_t)((e1_own - e0_own) * nranks * per_e * 4));
        landed = mbar_wait_cluster(red_bar, 0, p.status);
    }
    if (landed && *hdr_flag != 0) {
        if (GATED) {
            const int total = nrows * 64;
            const int share = (total + nranks - 1) / nranks;
            const int e0 = rank * share, e1 = min(total, e0 + share);
            for (int ei = e0 + tid; ei < e1; ei += kThreads) {
                float gsum = 0.0f, usum = 0.0f;
                for (int r = 0; r < nranks; ++r) {
                    gsum += part[(r * share + (ei - e0)) * 2 + 0];
                    usum += part[(r * share + (ei - e0)) * 2 + 1];
                }
                const int t = ei / 64, jj = ei % 64;
                if (t < nrows)
                    p.H[(int64_t)(r0 + t) * p.I + (int64_t)cgi * 64 + jj] = f32_to_act_bits<F16>(silu_f(gsum) * usum);
            }
        } else {
            const int total = nrows * 128;
            const int share = (total + nranks - 1) / nranks;
            const int e0 = rank * share, e1 = min(total, e0 + share);
            for (int ei = e0 + tid; ei < e1; ei += kThreads) {
                float sum = 0.0f;
                for (int r = 0; r < nranks; ++r) sum += part[r * share + (ei - e0)];
                const int t = ei / 128, row = ei % 128;
                const int64_t n = row_a + row;
                if (t < nrows && n < p.N) {
                    if (ONE == 2) {          // the layer output: sum over the slots of p_j * y_j
                        p.out[n] = f32_to_act_bits<F16>(sum);
                    } else if (p.act != 0) {        // non-gated FC1: h = RN(act(v)) in permuted row order
                        p.H[(int64_t)(r0 + t) * p.N + n] = f32_to_act_bits<F16>(plain_act(sum, p.act));
                    } else {
                        const int32_t slot = p.perm[r0 + t];
                        p.Yp[(int64_t)slot * p.N + n] = p.wts[slot] * sum;
                    }
                }
            }
        }
    }
}

// ----------------------------------------- persistent grouped streaming --
// With many work items the layer runs one wave of CTAs instead of one CTA per
// (item, column group): CTA b walks the units u = b, b + G, ... (G CTAs; u =
// item * ncg + column group, K whole), and its producer warp keeps the ring
// streaming across unit boundaries, so no unit pays for a launch, barrier
// set-up, ring fill or drain.  Each unit's magnitude table (its expert's
// global) goes through one of two table slots, so the next unit's table lands
// while the current one is still read.  No split: the gated experts' up rows
// meet their gate rows through shared memory, the others write from
// registers.  When the routing tables were written two launches back (FC2 after
// FC1), the producer reads its first unit and streams that unit's first weight
// stages and table before the programmatic-launch wait; only the activation
// copies wait for the preceding kernel.
// Stages of two 64-k blocks: with three CTAs per SM a ring of two large
// stages keeps about one stage per CTA in flight while the other is read,
// which left the consumers waiting on data at a third of the HBM rate; five
// (four) small stages keep three to four in flight in the same shared memory.
template <int MT> struct PersistRing;
template <> struct PersistRing<1> { using G = StreamRing<1, 5, 2>; };
template <> struct PersistRing<2> { using G = StreamRing<2, 4, 2>; };
template <> struct PersistRing<4> { using G = StreamRing<4, 3, 2>; };

struct PersistSmem {
    static constexpr size_t flags = 112;       // int[2]: the unit in table slot i passed its header check
    static constexpr size_t lut = 128;         // 2 slots x (1, or 2 with gate/up shards) tables
};

size_t persist_smem(int MT, bool gated, bool shards) {
    const int tok = 8 * MT;
    const size_t ring = MT == 1   ? PersistRing<1>::G::kStages * PersistRing<1>::G::kStageBytes
                        : MT == 2 ? PersistRing<2>::G::kStages * PersistRing<2>::G::kStageBytes
                                  : PersistRing<4>::G::kStages * PersistRing<4>::G::kStageBytes;
    const size_t part = gated ? (size_t)tok * 64 * 4 : 0;
    const size_t epi = (size_t)2 * tok * 8;        // FC2: routing slot and weight per row, per table slot
    return PersistSmem::lut + 2 * (shards ? 2 : 1) * kLutBytes + ring + part + epi;
}

template <int MT, bool GATED, bool F16, bool AWQ>
__global__ void __launch_bounds__(kThreads, 3)
moe_persist_kernel(const MoeLinParams p, int ncg, int early) {
    extern __shared__ __align__(128) uint8_t smem[];
    using G = typename PersistRing<MT>::G;
    constexpr int TOK = G::kTok;
    constexpr int kStages = G::kStages;
    constexpr int kBlocksPerStage = G::kBlocksPerStage;
    constexpr uint32_t kWeightStageBytes = G::kWeightStageBytes;
    constexpr int kXRowElems = G::kXRowElems;
    constexpr size_t kStageBytes = G::kStageBytes;
    static_assert((2 * kStages + 4) * 8 <= PersistSmem::flags, "barriers overlap the unit flags");
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStages;
    uint64_t* lut_full = empty + kStages;     // table slot i holds the current unit's table(s)
    uint64_t* lut_empty = lut_full + 2;       // every consumer warp is done with table slot i
    volatile int* unit_ok = reinterpret_cast<volatile int*>(smem + PersistSmem::flags);
    const bool shards = GATED && p.half_stride != 0;
    const int ntab = shards ? 2 : 1;
    uint4* lut = reinterpret_cast<uint4*>(smem + PersistSmem::lut);
    uint8_t* ring = smem + PersistSmem::lut + 2 * ntab * kLutBytes;
    float* part = reinterpret_cast<float*>(ring + kStages * kStageBytes);   // gated: up values [64][TOK]
    // FC2 epilogue operands of the unit in table slot i: routing slot and
    // routing weight of each row, written by the producer with the unit's table
    int32_t* ep_slot = reinterpret_cast<int32_t*>(part + (GATED ? 64 * TOK : 0));   // [2][TOK]
    float* ep_w = reinterpret_cast<float*>(ep_slot + 2 * TOK);                      // [2][TOK]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nst = (int)((p.KB + kBlocksPerStage - 1) / kBlocksPerStage);
    const int64_t stride = gridDim.x;
    // K is a multiple of 64 here: every k of a stage's blocks holds data
    auto stage_nb = [&](int i) { return (int)min((int64_t)kBlocksPerStage, p.KB - (int64_t)i * kBlocksPerStage); };
    auto stage_kx = [&](int i) { return (int64_t)i * kBlocksPerStage * kBlockK; };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&lut_full[i], 1);
            mbar_init(&lut_empty[i], kWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kWarps) {
        // ---------------- producer: the whole warp issues each stage's copies
        // (lane b a weight block or half-block, lane t activation row t) after
        // lane 0 has armed the stage's barrier; lane 0 alone waits on barriers
        // and the warp follows its verdict.
        const unsigned all = 0xffffffffu;
        // early: 0 = wait first; 1 = the first weight stages before the wait;
        // 2 = nothing read depends on the preceding kernel: wait only at the
        // end, so that this kernel completes after it
        bool waited = early == 0;
        const bool late = early == 2;
        if (waited) {
            pdl_wait_previous();
            pdl_launch_dependents();
        }
        const int64_t units = (int64_t)__ldcg(p.n_items) * ncg;
        const bool token_rows = GATED || p.act != 0;
        int gs = 0;                    // stages issued so far
        int j = 0;                     // units taken so far
        bool ok = true;
        for (int64_t u = blockIdx.x; u < units && ok; u += stride, ++j) {
            const int4 item = __ldcg(p.items + u / ncg);
            const int cgi = (int)(u % ncg);
            const int e = item.x, r0 = item.y, nrows = item.z;
            const uint8_t* wexp = p.w + (size_t)e * p.w_stride;
            const uint8_t* wup = shards ? wexp + p.half_stride : wexp;
            const int slot = j & 1;
            int hdr_ok = 0;
            if (lane == 0) {
                const Header* hdr = reinterpret_cast<const Header*>(wexp);
                const Header* hdr_up = reinterpret_cast<const Header*>(wup);
                hdr_ok = hdr->magic == kMagic && hdr->N == p.N && hdr->K == p.K &&
                         (!shards || (hdr_up->magic == kMagic && hdr_up->N == p.N && hdr_up->K == p.K));
                if (j >= 2) ok = mbar_wait(&lut_empty[slot], ((j >> 1) - 1) & 1, p.status);
                if (ok) {
                    unit_ok[slot] = hdr_ok;
                    if (!hdr_ok) {
                        record_status(p.status, NVFP4_ERR_BAD_WEIGHT);
                        mbar_arrive(&lut_full[slot]);          // the consumers skip this unit
                    } else {
                        uint4* ls = lut + slot * ntab * 256;
                        mbar_arrive_expect_tx(&lut_full[slot], (uint32_t)(ntab * kLutBytes));
                        bulk_g2s(ls, wexp + lut_offset<F16>(), (uint32_t)kLutBytes, &lut_full[slot]);
                        if (shards) bulk_g2s(ls + 256, wup + lut_offset<F16>(), (uint32_t)kLutBytes, &lut_full[slot]);
                    }
                }
            }
            ok = __shfl_sync(all, ok ? 1 : 0, 0) != 0;
            if (!ok) break;                            // unit j was not taken: j units were
            if (!__shfl_sync(all, hdr_ok, 0)) continue;
            // this lane's copies: weight block (or gate / up half-block) `lane`
            // of each stage, and activation row `lane`
            const int64_t row_a = GATED ? (int64_t)cgi * 64 : (int64_t)cgi * 128;
            const int64_t row_b = GATED ? (shards ? 0 : p.I) + (int64_t)cgi * 64 : 0;
            constexpr int kCopiesPerBlock = GATED ? 2 : 1;
            const int wb = lane / kCopiesPerBlock;                        // block within the stage
            const bool up_half = GATED && (lane & 1);
            const int64_t rbg = (up_half ? row_b : row_a) / kAtomRows;
            const uint8_t* wsrc = (up_half ? wup : wexp) + kTilesOffset +
                                  atom_offset(rbg / kAtomsPerTileK, 0, rbg % kAtomsPerTileK, p.KB);
            constexpr uint32_t kCopyBytes = kBlockBytes / kCopiesPerBlock;
            const size_t kb_stride = (size_t)kAtomsPerTileK * kAtomBytes;
            const uint16_t* xsrc = p.X;
            if (lane < nrows) {
                const int64_t r = r0 + lane;
                xsrc = p.X + (token_rows ? (int64_t)(__ldcg(p.perm + r) / p.topk) : r) * p.K;
                if (!token_rows) {
                    const int32_t sl = __ldcg(p.perm + r);
                    ep_slot[slot * TOK + lane] = sl;
                    ep_w[slot * TOK + lane] = __ldcg(p.wts + sl);
                }
            }
            __syncwarp();          // those writes before lane 0 arms the unit's first stage
            auto issue_weights = [&](int i, int s) {
                const int nb = stage_nb(i);
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[s], (uint32_t)(nb * kBlockBytes + (size_t)nrows * nb * kBlockK * 2));
                __syncwarp();
                if (wb < nb)
                    bulk_g2s(ring + s * kStageBytes + lane * kCopyBytes,
                             wsrc + (size_t)(i * kBlocksPerStage + wb) * kb_stride, kCopyBytes, &full[s]);
            };
            auto issue_x = [&](int i, int s) {
                if (lane < nrows)
                    bulk_g2s(ring + s * kStageBytes + kWeightStageBytes + lane * kXRowElems * 2,
                             xsrc + stage_kx(i), (uint32_t)(stage_nb(i) * kBlockK * 2), &full[s]);
            };
            int i = 0;
            if (!waited && !late) {
                // weights (and the table, above) before the wait, activations
                // after it; no stage has been issued yet (gs == 0)
                const int pre = min(nst, kStages);
                for (; i < pre; ++i) issue_weights(i, i);
                pdl_wait_previous();
                pdl_launch_dependents();
                waited = true;
                for (int k = 0; k < pre; ++k) issue_x(k, k);
                gs = pre;
            }
            for (; i < nst; ++i, ++gs) {
                const int s = gs % kStages;
                if (gs >= kStages) {
                    bool got = true;
                    if (lane == 0) got = mbar_wait(&empty[s], ((gs / kStages) - 1) & 1, p.status);
                    if (!(ok = __shfl_sync(all, got ? 1 : 0, 0) != 0)) break;
                }
                issue_weights(i, s);
                issue_x(i, s);
            }
        }
        if (!waited) {
            pdl_wait_previous();
            pdl_launch_dependents();
        }
        // never leave a copy in flight into this CTA's shared memory
        if (lane == 0) {
            for (int k = max(0, j - 2); k < j; ++k) mbar_wait(&lut_full[k & 1], (k >> 1) & 1, p.status);
            for (int k = max(0, gs - kStages); k < gs; ++k) mbar_wait(&full[k % kStages], (k / kStages) & 1, p.status);
        }
        __syncwarp();
    } else {
        // ---------------- consumers
        if (early != 2) {
            pdl_wait_previous();
            pdl_launch_dependents();
        }
        const int g = lane >> 2, q = lane & 3, c = lane & 3;
        const int64_t units = (int64_t)(*p.n_items) * ncg;
        const uint8_t* const a0 = ring + warp * kAtomBytes;
        const uint16_t* const x0 = reinterpret_cast<const uint16_t*>(ring + kWeightStageBytes) +
                                   g * kXRowElems + q * 16;
        using AwqStagesT = AwqStages<F16, kXRowElems, TOK, kBlocksPerStage, kWarps * 32>;
        AwqStagesT awq;
        // every unit walks the same k stages: the scales of stage i are unit-independent
        if constexpr (AWQ) awq.prefetch(p.pqs, TOK, stage_nb(0) * kBlockK, tid);
        int s = 0;
        uint32_t phase = 0;
        int j = 0;
        int4 item = (int64_t)blockIdx.x < units ? p.items[blockIdx.x / ncg] : make_int4(0, 0, 0, 0);
        for (int64_t u = blockIdx.x; u < units; u += stride, ++j) {
            const int slot = j & 1;
            const int cgi = (int)(u % ncg);
            const int r0 = item.y, nrows = item.z;
            // the next unit's item loads while this unit's stages stream
            if (u + stride < units) item = p.items[(u + stride) / ncg];
            // every consumer warp leaves together when one could not go on
            if (!named_bar_red_and(1, kWarps * 32, mbar_wait(&lut_full[slot], (j >> 1) & 1, p.status))) break;
            const bool valid = unit_ok[slot] != 0;
            const int64_t row_a = GATED ? (int64_t)cgi * 64 : (int64_t)cgi * 128;
            const bool rows_valid = GATED || row_a + warp * kAtomRows < p.N;
            const uint32_t lut_s = smem_u32(lut + slot * ntab * 256 + ((shards && warp >= 4) ? 256 : 0));
            float acc[MT][4];
            #pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                #pragma unroll
                for (int v = 0; v < 4; ++v) acc[mt][v] = 0.0f;
            bool ok = true;
            if (valid) {
                for (int i = 0; i < nst; ++i) {
                    const bool got = mbar_wait(&full[s], phase, p.status);
                    if constexpr (!AWQ) {
                        if (!got) { ok = false; break; }
                    } else {
                        AwqStagesT nxt = awq;
                        const int in = i + 1 < nst ? i + 1 : 0;
                        nxt.prefetch(p.pqs + stage_kx(in), TOK, stage_nb(in) * kBlockK, tid);
                        if (got)
                            awq.apply(reinterpret_cast<uint16_t*>(ring + s * kStageBytes + kWeightStageBytes), nrows,
                                      stage_nb(i) * kBlockK, tid);
                        awq = nxt;
                        if (!named_bar_red_and(1, kWarps * 32, got)) { ok = false; break; }
                    }
                    if (rows_valid)
                        stage_mma<MT, kXRowElems, F16, kBlocksPerStage, kBlockBytes>(
                            a0 + s * kStageBytes, lane, lut_s, x0 + s * (kStageBytes / 2), stage_nb(i), acc,
                            MT == 1 ? 1 : (nrows + 7) >> 3);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    if (++s == kStages) { s = 0; phase ^= 1u; }
                }
            }
            if (!named_bar_red_and(1, kWarps * 32, ok)) break;
            if (valid) {
            if constexpr (GATED) {
                // up rows (warps 4-7) hand their values to the gate rows (warps 0-3)
                if (warp >= 4) {
                    #pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        #pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int jj = (warp - 4) * 16 + g + (v >= 2 ? 8 : 0);
                            part[jj * TOK + mt * 8 + 2 * c + (v & 1)] = acc[mt][v];
                        }
                }
                named_bar_sync(2, kWarps * 32);
                if (warp < 4) {
                    #pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
                        #pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int jj = warp * 16 + g + (v >= 2 ? 8 : 0);
                            const int t = mt * 8 + 2 * c + (v & 1);
                            if (t < nrows)
                                p.H[(int64_t)(r0 + t) * p.I + (int64_t)cgi * 64 + jj] =
                                    f32_to_act_bits<F16>(silu_f(acc[mt][v]) * part[jj * TOK + t]);
                        }
                }
                named_bar_sync(2, kWarps * 32);
            } else {
                #pragma unroll
                for (int mt = 0; mt < MT; ++mt)
                    #pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int t = mt * 8 + 2 * c + (v & 1);
                        const int64_t n = row_a + warp * 16 + g + (v >= 2 ? 8 : 0);
                        if (t < nrows && n < p.N) {
                            if (p.act != 0)
                                p.H[(int64_t)(r0 + t) * p.N + n] = f32_to_act_bits<F16>(plain_act(acc[mt][v], p.act));
                            else
                                p.Yp[(int64_t)ep_slot[slot * TOK + t] * p.N + n] = ep_w[slot * TOK + t] * acc[mt][v];
                        }
                    }
            }
            }
            // the table slot (and its epilogue operands) may be refilled
            __syncwarp();
            if (lane == 0) mbar_arrive(&lut_empty[slot]);
        }
    }
}

// ----------------------------------------------------------------- combine --
template <bool F16>
__global__ void combine_kernel(const float* __restrict__ Yp, int64_t T, int topk, int64_t H,
                               uint16_t* __restrict__ out) {
    pdl_wait_previous();
    pdl_launch_dependents();
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= T * H) return;
    const int64_t t = i / H, n = i % H;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < topk; ++j) {
        const float4 v = *reinterpret_cast<const float4*>(Yp + (t * topk + j) * H + n);
        s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    const uint32_t lo = (uint32_t)f32_to_act_bits<F16>(s.x) | ((uint32_t)f32_to_act_bits<F16>(s.y) << 16);
    const uint32_t hi = (uint32_t)f32_to_act_bits<F16>(s.z) | ((uint32_t)f32_to_act_bits<F16>(s.w) << 16);
    *reinterpret_cast<uint2*>(out + i) = make_uint2(lo, hi);
}

// Rows of X in permuted (expert-contiguous) order, for the tile path:
// Xp[r] = X[perm[r] / topk], times the AWQ pre-quant scale when given.  A
// thread moves kGatherChunks 16-byte chunks, blockDim chunks apart, with all
// their row-index loads and then all their data loads in flight at once.
constexpr int kGatherChunks = 4;

template <bool F16>
__global__ void gather_rows_kernel(const uint16_t* __restrict__ X, const uint16_t* __restrict__ pqs,
                                   const int32_t* __restrict__ perm, int topk, int64_t n, int64_t H,
                                   uint16_t* __restrict__ Xp) {
    pdl_wait_previous();
    pdl_launch_dependents();
    const int64_t chunks = n * H / 8;
    const int64_t c0 = (int64_t)blockIdx.x * blockDim.x * kGatherChunks + threadIdx.x;
    int64_t src[kGatherChunks];
    #pragma unroll
    for (int u = 0; u < kGatherChunks; ++u) {
        const int64_t i = (c0 + (int64_t)u * blockDim.x) * 8;
        src[u] = i < n * H ? (int64_t)(perm[i / H] / topk) * H + i % H : -1;
    }
    uint4 v[kGatherChunks];
    #pragma unroll
    for (int u = 0; u < kGatherChunks; ++u)
        if (src[u] >= 0) v[u] = *reinterpret_cast<const uint4*>(X + src[u]);
    #pragma unroll
    for (int u = 0; u < kGatherChunks; ++u) {
        const int64_t c = c0 + (int64_t)u * blockDim.x;
        if (c >= chunks) continue;
        if (pqs != nullptr) {
            const uint4 sv4 = *reinterpret_cast<const uint4*>(pqs + (c * 8) % H);
            uint32_t xv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            const uint32_t sv[4] = {sv4.x, sv4.y, sv4.z, sv4.w};
            #pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint16_t lo = awq_mul<F16>((uint16_t)(xv[e] & 0xFFFF), (uint16_t)(sv[e] & 0xFFFF));
                const uint16_t hi = awq_mul<F16>((uint16_t)(xv[e] >> 16), (uint16_t)(sv[e] >> 16));
                xv[e] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            v[u] = make_uint4(xv[0], xv[1], xv[2], xv[3]);
        }
        *reinterpret_cast<uint4*>(Xp + c * 8) = v[u];
    }
}

// Launch with programmatic dependent launch enabled (see route_kernel).
template <typename... Params, typename... Args>
nvfp4_status launch_chained(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            const char* what, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return check_cuda(cudaLaunchKernelEx(&cfg, kernel, args...), what);
}

size_t moe_lin_smem(int MT, bool gated, bool shards) {
    const int tok = 8 * MT;
    const size_t part = gated ? ((size_t)tok * 64 + 8) * 2 : (size_t)tok * 128 + 8;
    const size_t ring = MT == 1   ? MoeRing<1>::G::kStages * MoeRing<1>::G::kStageBytes
                        : MT == 2 ? MoeRing<2>::G::kStages * MoeRing<2>::G::kStageBytes
                                  : MoeRing<4>::G::kStages * MoeRing<4>::G::kStageBytes;
    return kRingOffset + (shards ? 2 : 1) * kLutBytes + ring + part * 4;
}

template <int MT, bool GATED, bool F16, bool AWQ>
nvfp4_status launch_moe_linear_typed(const MoeLinParams& p, unsigned gx, unsigned max_items, cudaStream_t s) {
    const size_t smem = moe_lin_smem(MT, GATED, GATED && p.half_stride != 0);
    cudaError_t e = cudaFuncSetAttribute(moe_linear_kernel<MT, GATED, F16, AWQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return check_cuda(e, "MoE linear: shared memory attribute");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, (unsigned)p.splits, max_items);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)p.splits;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, moe_linear_kernel<MT, GATED, F16, AWQ>, p);
    return check_cuda(e, GATED ? "MoE FC1: launch" : "MoE FC2: launch");
}

// Resident CTAs per SM of a persistent instance (registers, shared memory and
// threads), looked up once per instance.
template <int MT, bool GATED, bool F16, bool AWQ>
int persist_ctas_per_sm(size_t smem) {
    static int cache[2] = {0, 0};
    static std::once_flag once[2];
    const int k = smem > persist_smem(MT, GATED, false) ? 1 : 0;      // with gate/up shards
    std::call_once(once[k], [&] {
        int n = 0;
        if (cudaFuncSetAttribute(moe_persist_kernel<MT, GATED, F16, AWQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, moe_persist_kernel<MT, GATED, F16, AWQ>, kThreads,
                                                          smem) == cudaSuccess)
            cache[k] = n;
    });
    return cache[k];
}

template <int MT, bool GATED, bool F16, bool AWQ>
nvfp4_status launch_moe_persist_typed(const MoeLinParams& p, int ncg, int64_t max_units, int early, cudaStream_t s) {
    const size_t smem = persist_smem(MT, GATED, GATED && p.half_stride != 0);
    cudaError_t e = cudaFuncSetAttribute(moe_persist_kernel<MT, GATED, F16, AWQ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return check_cuda(e, "MoE persistent linear: shared memory attribute");
    const int per_sm = std::max(1, persist_ctas_per_sm<MT, GATED, F16, AWQ>(smem));
    const int64_t grid = std::min<int64_t>(max_units, (int64_t)per_sm * sm_count());
    return launch_chained(moe_persist_kernel<MT, GATED, F16, AWQ>, dim3((unsigned)std::max<int64_t>(grid, 1)),
                          dim3(kThreads), smem, s, GATED ? "MoE FC1 (persistent): launch" : "MoE FC2 (persistent): launch",
                          p, ncg, early);
}

// The persistent instance for the activation type and AWQ choice.
template <int MT, bool GATED>
nvfp4_status launch_moe_persist(const MoeLinParams& p, int ncg, int64_t max_units, int early, bool f16,
                                cudaStream_t s) {
    if (p.pqs != nullptr)
        return f16 ? launch_moe_persist_typed<MT, GATED, true, true>(p, ncg, max_units, early, s)
                   : launch_moe_persist_typed<MT, GATED, false, true>(p, ncg, max_units, early, s);
    return f16 ? launch_moe_persist_typed<MT, GATED, true, false>(p, ncg, max_units, early, s)
               : launch_moe_persist_typed<MT, GATED, false, false>(p, ncg, max_units, early, s);
}

template <int MT, bool GATED>
nvfp4_status launch_moe_linear(const MoeLinParams& p, unsigned gx, unsigned max_items, bool f16, cudaStream_t s) {
    // AWQ instances: FC1 with a pre-quant scale on its input
    if (p.pqs != nullptr)
        return f16 ? launch_moe_linear_typed<MT, GATED, true, true>(p, gx, max_items, s)
                   : launch_moe_linear_typed<MT, GATED, false, true>(p, gx, max_items, s);
    return f16 ? launch_moe_linear_typed<MT, GATED, true, false>(p, gx, max_items, s)
               : launch_moe_linear_typed<MT, GATED, false, false>(p, gx, max_items, s);
}

// Single-token kernels: FC1 (ONE = 1; K split across a cluster of `splits`)
// and FC2 with the combine (ONE = 2; one cluster per row group over the topk
// slots and their `splits` K splits), both with grid z = the routing slot.
template <bool GATED, bool F16, bool AWQ, int ONE>
nvfp4_status launch_moe_one_typed(const MoeLinParams& p, unsigned gx, cudaStream_t s) {
    const size_t smem = moe_lin_smem(1, GATED, GATED && p.half_stride != 0);
    cudaError_t e = cudaFuncSetAttribute(moe_linear_kernel<1, GATED, F16, AWQ, ONE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return check_cuda(e, "MoE single token: shared memory attribute");
    const unsigned ys = (unsigned)p.splits;
    const unsigned zs = ONE == 2 ? (unsigned)p.topk : 1u;
    if (ys * zs > 8) {             // clusters of up to 16 CTAs are not portable: opt in
        e = cudaFuncSetAttribute(moe_linear_kernel<1, GATED, F16, AWQ, ONE>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return check_cuda(e, "MoE single token: cluster size attribute");
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, ys, (unsigned)p.topk);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = ys;
    attr[0].val.clusterDim.z = zs;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, moe_linear_kernel<1, GATED, F16, AWQ, ONE>, p);
    return check_cuda(e, ONE == 1 ? "MoE single-token FC1: launch" : "MoE single-token FC2: launch");
}

// The instances for 8, 16 or 32 routed rows per work item.
template <bool GATED>
nvfp4_status launch_moe_linear_mt(int mt, const MoeLinParams& p, unsigned gx, unsigned max_items, bool f16,
                                  cudaStream_t s) {
    return mt == 1   ? launch_moe_linear<1, GATED>(p, gx, max_items, f16, s)
           : mt == 2 ? launch_moe_linear<2, GATED>(p, gx, max_items, f16, s)
                     : launch_moe_linear<4, GATED>(p, gx, max_items, f16, s);
}

template <bool GATED>
nvfp4_status launch_moe_persist_mt(int mt, const MoeLinParams& p, int ncg, int64_t max_units, int early, bool f16,
                                   cudaStream_t s) {
    return mt == 1   ? launch_moe_persist<1, GATED>(p, ncg, max_units, early, f16, s)
           : mt == 2 ? launch_moe_persist<2, GATED>(p, ncg, max_units, early, f16, s)
                     : launch_moe_persist<4, GATED>(p, ncg, max_units, early, f16, s);
}

// Tile path: an expert's last few rows past its full tiles (at most this many)
// run as one 32-row item of the streaming kernels instead of a whole tile.
constexpr int kTileTailRows = 32;

struct MoeLayout {
    size_t idx, wts, offsets, perm, inv, items, n_items, counts, xp, h, yp, total;
    bool tile;              // tensor-core tile path (many rows per expert) or the streaming path
    int tok, mt, subm;
    int tail_rows;          // tile path: kTileTailRows (tail items follow the max_items main ones)
    int64_t max_items;
};

MoeLayout moe_layout(int64_t T, int E, int topk, int64_t H, int64_t I) {
    MoeLayout L{};
    const int64_t n = T * topk;
    const int64_t per_expert = n / std::max(E, 1);   // routed rows per expert on average
    // Many rows per expert: tcgen05 tiles of 128 (or 256) routed rows; fewer:
    // the streaming kernel with 8 or 16 rows per work item.  At 16 to 31 rows
    // per expert the streaming kernel, which expands weights on far more warps
    // than the tile kernel has, measured faster despite reading an expert
    // twice when its rows need two items.
    L.tile = per_expert >= 32 && I % 128 == 0;
    L.subm = per_expert >= 192 ? 2 : 1;
    // rows per streaming item: 8, 16 or 32 -- at 13 or more rows per expert on
    // average 32-row items hold most experts whole, so that their weights are
    // expanded once instead of once per 16 rows
    L.mt = per_expert > 12 ? 4 : per_expert > 8 ? 2 : 1;
    L.tok = L.tile ? 128 * L.subm : 8 * L.mt;
    L.max_items = ceil_div(n, L.tok) + std::min<int64_t>(E, n);
    size_t off = 0;
    auto take = [&](size_t bytes) { const size_t o = off; off += (size_t)round_up((int64_t)bytes, 256); return o; };
    L.idx = take(n * 4);
    L.wts = take(n * 4);
    L.offsets = take((E + 1) * 4);
    L.perm = take(n * 4);
    L.inv = take(n * 4);
    L.tail_rows = L.tile ? kTileTailRows : 0;
    L.items = take((L.max_items + (L.tile ? E : 0)) * 16);
    L.n_items = take(8);
    L.counts = T >= kChunkedRouteMinT ? take((size_t)E * (route_chunks(T) + 1) * 4) : 0;
    L.xp = L.tile ? take(n * H * 2) : 0;
    L.h = take(n * I * 2);
    L.yp = take(n * H * 4);
    L.total = off;
    return L;
}

// Route (top-k + softmax over the selected logits) and permute (counts,
// offsets, stable permutation, its inverse, and -- when `items` is not null --
// the work list of `tok`-row items): one fused single-CTA kernel for few
// tokens; else, with `counts` scratch (E x (ceil(T / 8) + 1) ints), the three
// chunked kernels; without it a routing kernel and a single-CTA permutation.
nvfp4_status launch_routing(const float* router_logits, int64_t T, int E, int topk, int tok, int32_t* idx,
                            float* wts, int32_t* offsets, int32_t* perm, int32_t* inv, int4* items,
                            int32_t* n_items, cudaStream_t s, int32_t* counts = nullptr, int tail_rows = 0,
                            int tail_base = 0) {
    nvfp4_status st;
    const int wc = permute_words(T, E, topk);
    const size_t psmem = permute_smem_bytes(E, wc);
    if (T <= kFusedRouteMaxT)
        return launch_chained(route_permute_kernel, dim3(1), dim3(kPermThreads), 0, s, "MoE route+permute: launch",
                              router_logits, T, E, topk, tok, idx, wts, offsets, perm, inv, items, n_items,
                              tail_rows, tail_base);
    if (counts != nullptr) {
        const int C = (int)route_chunks(T);
        int32_t* totals = counts + (int64_t)E * C;
        st = launch_chained(route_count_kernel, dim3((unsigned)C), dim3(kChunkThreads), 0, s,
                            "MoE route+count: launch", router_logits, T, E, topk, idx, wts, counts, C);
        if (st != NVFP4_OK) return st;
        st = launch_chained(chunk_scan_kernel, dim3((unsigned)ceil_div(E, kScanWarps)), dim3(kScanWarps * 32), 0, s,
                            "MoE chunk scan: launch", counts, C, E, totals);
        if (st != NVFP4_OK) return st;
        return launch_chained(chunk_permute_kernel, dim3((unsigned)C), dim3(kChunkTokens * kMaxTopk), 0, s,
                              "MoE chunk permute: launch", (const int32_t*)idx, T, topk, E, tok,
                              (const int32_t*)counts, (const int32_t*)totals, C, offsets, perm, inv, items,
                              n_items, tail_rows, tail_base);
    }
    st = launch_chained(route_kernel, dim3((unsigned)ceil_div(T, 8)), dim3(256), 0, s, "MoE route: launch",
                        router_logits, T, E, topk, idx, wts);
    if (st != NVFP4_OK) return st;
    cudaError_t ce = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
    if ((st = check_cuda(ce, "MoE permute: shared memory attribute")) != NVFP4_OK) return st;
    return launch_chained(permute_kernel, dim3(1), dim3(kPermThreads), psmem, s, "MoE permute: launch",
                          (const int32_t*)idx, T, topk, E, tok, wc, offsets, perm, inv, items, n_items, tail_rows,
                          tail_base);
}

// Work items expected in flight, for the split-K and persistent choices of the
// streaming path (the exact count is known only on the device).
int64_t moe_est_items(const MoeLayout& L, int64_t n, int E) {
    return std::min<int64_t>(L.max_items, std::max<int64_t>(ceil_div(n, L.tok), std::min<int64_t>(E, n)));
}

// Units (item x column group) for several waves: one persistent wave walks
// them without splitting K; fewer: a CTA per unit, K split across a cluster.
bool moe_use_persist(int64_t fc1_groups, int64_t est_items) { return fc1_groups * est_items >= 4LL * sm_count(); }

// One token whose top-k fits one portable cluster: the two single-token kernels.
bool moe_single_token(int64_t T, int topk) { return T == 1 && topk <= 8; }

int moe_splits(int64_t base_ctas, int64_t KB, int kbs_min) {
    int64_t splits = std::max<int64_t>(1, ceil_div(2LL * sm_count(), std::max<int64_t>(base_ctas, 1)));
    splits = std::min<int64_t>(splits, std::min<int64_t>(8, std::max<int64_t>(1, KB / kbs_min)));
    return (int)splits;
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_moe_route(const float* router_logits, int64_t T, int E, int topk,
                                       int32_t* topk_idx_out, float* topk_weight_out, int32_t* perm_out,
                                       int32_t* inv_out, int32_t* offsets_out, void* stream) {
    const char* fn = "nvfp4_moe_route";
    if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "%s: T=%lld is negative", fn, (long long)T);
    if (E < 1 || E > kMaxExperts) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: E=%d outside [1, %d]", fn, E, kMaxExperts);
    if (topk < 1 || topk > kMaxTopk || topk > E) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: topk=%d outside [1, min(E, %d)]", fn, topk, kMaxTopk);
    if (T * topk >= ((int64_t)1 << 31)) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: T*topk=%lld exceeds int32 slots", fn, (long long)(T * topk));
    if (T == 0) return NVFP4_OK;                  // a zero-token chunk launches no kernel
    if (!router_logits || !topk_idx_out || !topk_weight_out || !perm_out || !inv_out || !offsets_out)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(router_logits, 4) || !aligned(topk_idx_out, 4) || !aligned(topk_weight_out, 4) ||
        !aligned(perm_out, 4) || !aligned(inv_out, 4) || !aligned(offsets_out, 4))
        return fail(NVFP4_ERR_ALIGNMENT, "%s: every pointer must be 4-byte aligned", fn);
    return launch_routing(router_logits, T, E, topk, 1, topk_idx_out, topk_weight_out, offsets_out, perm_out,
                          inv_out, nullptr, nullptr, (cudaStream_t)stream);
}

extern "C" nvfp4_status nvfp4_w4a16_moe_plan(int64_t T, int E, int topk, int64_t H, int64_t I, int activation,
                                             int* path_out, int* rows_per_item_out) {
    const char* fn = "nvfp4_w4a16_moe_plan";
    if (!path_out || !rows_per_item_out) return fail(NVFP4_ERR_INVALID_ARG, "%s: null output pointer", fn);
    if (activation < NVFP4_MOE_SWIGLU || activation > NVFP4_MOE_SILU)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: activation=%d is not one of SWIGLU, RELU2, SILU", fn, activation);
    if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "%s: T=%lld is negative", fn, (long long)T);
    if (E < 1 || E > kMaxExperts) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: E=%d outside [1, %d]", fn, E, kMaxExperts);
    if (topk < 1 || topk > kMaxTopk || topk > E) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: topk=%d outside [1, min(E, %d)]", fn, topk, kMaxTopk);
    if (H <= 0 || I <= 0 || H % 64 != 0 || I % 64 != 0)
        return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: H=%lld and I=%lld must be positive multiples of 64", fn, (long long)H, (long long)I);
    if (T == 0) {
        *path_out = 0;
        *rows_per_item_out = 0;
        return NVFP4_OK;
    }
    const MoeLayout L = moe_layout(T, E, topk, H, I);
    const int64_t fc1_groups = activation == NVFP4_MOE_SWIGLU ? I / 64 : ceil_div(I, 128);
    *path_out = moe_single_token(T, topk) ? 4
              : L.tile ? 3 : moe_use_persist(fc1_groups, moe_est_items(L, T * topk, E)) ? 2 : 1;
    *rows_per_item_out = L.tok;
    return NVFP4_OK;
}

extern "C" size_t nvfp4_w4a16_moe_workspace(int64_t T, int E, int topk, int64_t H, int64_t I) {
    if (T <= 0 || E <= 0 || topk <= 0 || H <= 0 || I <= 0) return 0;
    return moe_layout(T, E, topk, H, I).total;
}

namespace nvfp4 {
namespace {

nvfp4_status moe_impl(const void* X, const float* router_logits, const void* fc1, const void* fc2,
                      const void* fc1_pre_quant_scale, int64_t T, int E, int topk, int64_t H, int64_t I,
                      int activation, int fc1_split, void* out, int32_t* topk_idx_out, float* topk_weight_out,
                      int32_t* perm_out, int32_t* offsets_out, void* workspace, size_t workspace_bytes, bool f16,
                      void* stream) {
    const bool ex = activation != NVFP4_MOE_SWIGLU || fc1_split != 0;
    const char* fn = ex ? "nvfp4_w4a16_moe_grouped_ex" : f16 ? "nvfp4_w4a16_moe_grouped_f16" : "nvfp4_w4a16_moe_grouped";
    if (activation < NVFP4_MOE_SWIGLU || activation > NVFP4_MOE_SILU)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: activation=%d is not one of SWIGLU, RELU2, SILU", fn, activation);
    if (fc1_split != 0 && (fc1_split != 1 || activation != NVFP4_MOE_SWIGLU))
        return fail(NVFP4_ERR_INVALID_ARG, "%s: fc1_split=%d (1 only with the gated SWIGLU experts)", fn, fc1_split);
    if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "%s: T=%lld is negative", fn, (long long)T);
    if (E < 1 || E > kMaxExperts) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: E=%d outside [1, %d]", fn, E, kMaxExperts);
    if (topk < 1 || topk > kMaxTopk || topk > E) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: topk=%d outside [1, min(E, %d)]", fn, topk, kMaxTopk);
    if (H <= 0 || I <= 0 || H % 64 != 0 || I % 64 != 0)
        return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: H=%lld and I=%lld must be positive multiples of 64", fn, (long long)H, (long long)I);
    if (T == 0) return NVFP4_OK;                  // a zero-token chunk launches no kernel
    if (!X || !router_logits || !fc1 || !fc2 || !out) return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(X, 16) || !aligned(out, 16)) return fail(NVFP4_ERR_ALIGNMENT, "%s: X and out must be 16-byte aligned", fn);
    if (!aligned(router_logits, 4)) return fail(NVFP4_ERR_ALIGNMENT, "%s: router_logits must be 4-byte aligned", fn);
    if (!aligned(fc1, 256) || !aligned(fc2, 256)) return fail(NVFP4_ERR_ALIGNMENT, "%s: expert weights must be 256-byte aligned", fn);
    if (fc1_pre_quant_scale && !aligned(fc1_pre_quant_scale, 16)) return fail(NVFP4_ERR_ALIGNMENT, "%s: fc1_pre_quant_scale must be 16-byte aligned", fn);
    if (moe_layout(T, E, topk, H, I).max_items > 65535)
        return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: T=%lld routes too many rows for one call", fn, (long long)T);
    const size_t need = nvfp4_w4a16_moe_workspace(T, E, topk, H, I);
    if (!workspace || workspace_bytes < need) return fail(NVFP4_ERR_WORKSPACE, "%s: workspace %zu bytes, needs %zu", fn, workspace_bytes, need);
    if (!aligned(workspace, 256)) return fail(NVFP4_ERR_ALIGNMENT, "%s: workspace must be 256-byte aligned", fn);
    int* status = device_status_ptr();
    if (!status) return fail(NVFP4_ERR_CUDA, "%s: no CUDA device", fn);

    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* ws = (uint8_t*)workspace;
    const MoeLayout L = moe_layout(T, E, topk, H, I);
    const int64_t n = T * topk;
    int32_t* idx = topk_idx_out ? topk_idx_out : (int32_t*)(ws + L.idx);
    float* wts = topk_weight_out ? topk_weight_out : (float*)(ws + L.wts);
    int32_t* offsets = offsets_out ? offsets_out : (int32_t*)(ws + L.offsets);
    int32_t* perm = perm_out ? perm_out : (int32_t*)(ws + L.perm);
    int32_t* inv = (int32_t*)(ws + L.inv);
    int4* items = (int4*)(ws + L.items);
    int32_t* n_items = (int32_t*)(ws + L.n_items);
    uint16_t* hbuf = (uint16_t*)(ws + L.h);
    float* yp = (float*)(ws + L.yp);
    nvfp4_status st;
    // FC1 of one expert: gated [2I, H] (gate rows, then up rows), or gate and up
    // shards [I, H] each with its own global, or non-gated [I, H]
    const bool gated = activation == NVFP4_MOE_SWIGLU;
    const size_t shard_bytes = nvfp4_repack_size(I, H);
    const size_t fc1_stride = !gated ? shard_bytes : fc1_split ? 2 * shard_bytes : nvfp4_repack_size(2 * I, H);
    const size_t half_stride = fc1_split ? shard_bytes : 0;
    const int64_t fc1_rows = (gated && !fc1_split) ? 2 * I : I;          // rows of one repacked FC1 buffer

    if (moe_single_token(T, topk)) {
        // One token: two kernels.  Every CTA routes the token itself; FC1 writes
        // h_j per slot, FC2 sums p_j * y_j over a cluster of the slots.
        MoeLinParams p1{};
        p1.w = (const uint8_t*)fc1; p1.w_stride = fc1_stride; p1.half_stride = half_stride;
        p1.N = fc1_rows; p1.K = H; p1.KB = round_up(H, kBlockK) / kBlockK;
        const int64_t fc1_groups = gated ? I / 64 : ceil_div(I, 128);
        p1.splits = moe_splits(fc1_groups * topk, p1.KB, 4);
        p1.kbs = (int)ceil_div(p1.KB, p1.splits);
        p1.splits = (int)ceil_div(p1.KB, p1.kbs);
        p1.X = (const uint16_t*)X; p1.topk = topk; p1.I = I; p1.H = hbuf; p1.status = status;
        p1.pqs = (const uint16_t*)fc1_pre_quant_scale;
        p1.act = gated ? 0 : activation;
        p1.logits = router_logits; p1.E = E;
        p1.r_idx = idx; p1.r_wts = wts; p1.r_perm = perm; p1.r_inv = inv; p1.r_offsets = offsets;
        const bool awq = fc1_pre_quant_scale != nullptr;
        if (gated)
            st = f16 ? (awq ? launch_moe_one_typed<true, true, true, 1>(p1, (unsigned)fc1_groups, s)
                            : launch_moe_one_typed<true, true, false, 1>(p1, (unsigned)fc1_groups, s))
                     : (awq ? launch_moe_one_typed<true, false, true, 1>(p1, (unsigned)fc1_groups, s)
                            : launch_moe_one_typed<true, false, false, 1>(p1, (unsigned)fc1_groups, s));
        else
            st = f16 ? (awq ? launch_moe_one_typed<false, true, true, 1>(p1, (unsigned)fc1_groups, s)
                            : launch_moe_one_typed<false, true, false, 1>(p1, (unsigned)fc1_groups, s))
                     : (awq ? launch_moe_one_typed<false, false, true, 1>(p1, (unsigned)fc1_groups, s)
                            : launch_moe_one_typed<false, false, false, 1>(p1, (unsigned)fc1_groups, s));
        if (st != NVFP4_OK) return st;
        MoeLinParams p2{};
        p2.w = (const uint8_t*)fc2; p2.w_stride = nvfp4_repack_size(H, I);
        p2.N = H; p2.K = I; p2.KB = round_up(I, kBlockK) / kBlockK;
        // K split in two when the slots' cluster stays within 16 CTAs: twice
        // the CTAs for FC2's small grid (one per row group and slot)
        const int64_t sp2 = (2 * topk <= 16 && p2.KB >= 4) ? 2 : 1;
        p2.kbs = (int)ceil_div(p2.KB, sp2);
        p2.splits = (int)ceil_div(p2.KB, (int64_t)p2.kbs);
        p2.X = hbuf; p2.topk = topk; p2.I = I; p2.status = status;
        p2.logits = router_logits; p2.E = E; p2.out = (uint16_t*)out;
        const unsigned fc2_groups = (unsigned)ceil_div(H, 128);
        return f16 ? launch_moe_one_typed<false, true, false, 2>(p2, fc2_groups, s)
                   : launch_moe_one_typed<false, false, false, 2>(p2, fc2_groups, s);
    }

    // AWQ: the tile path scales the rows while gathering them, the streaming
    // path the activation fragments inside FC1; no separate pass either way
    st = launch_routing(router_logits, T, E, topk, L.tok, idx, wts, offsets, perm, inv, items, n_items, s,
                        T >= kChunkedRouteMinT ? (int32_t*)(ws + L.counts) : nullptr, L.tail_rows,
                        (int)L.max_items);
    if (st != NVFP4_OK) return st;

    if (L.tile) {
        // gather the routed rows into expert-contiguous order, then two tile GEMMs
        uint16_t* xp = (uint16_t*)(ws + L.xp);
        st = launch_chained(f16 ? gather_rows_kernel<true> : gather_rows_kernel<false>,
                            dim3((unsigned)ceil_div(n * H / 8, 256 * kGatherChunks)), dim3(256), 0, s,
                            "MoE gather: launch", (const uint16_t*)X, (const uint16_t*)fc1_pre_quant_scale,
                            (const int32_t*)perm, topk, n, H, xp);
        if (st != NVFP4_OK) return st;
        TcMoeParams t1{};
        t1.fc1 = true; t1.f16 = f16; t1.subm = L.subm; t1.X = xp; t1.x_rows = n;
        t1.act = gated ? 0 : activation; t1.half_stride = half_stride;
        t1.w = (const uint8_t*)fc1; t1.w_stride = fc1_stride;
        t1.N = fc1_rows; t1.K = H; t1.I = I; t1.items = items; t1.n_items = n_items; t1.max_items = L.max_items;
        t1.perm = perm; t1.wts = wts; t1.H = hbuf; t1.status = status;
        if ((st = launch_tc_moe(t1, s)) != NVFP4_OK) return st;
        // the experts' tails (<= 32 rows past their last full tile): one wave of
        // the streaming kernel over the second item list, writing the same H rows
        int4* tails = items + L.max_items;
        int32_t* n_tails = n_items + 1;
        MoeLinParams q1{};
        q1.w = (const uint8_t*)fc1; q1.w_stride = fc1_stride; q1.half_stride = half_stride;
        q1.N = fc1_rows; q1.K = H; q1.KB = round_up(H, kBlockK) / kBlockK;
        q1.splits = 1; q1.kbs = (int)q1.KB;
        q1.X = (const uint16_t*)X; q1.perm = perm; q1.topk = topk; q1.items = tails; q1.n_items = n_tails;
        q1.I = I; q1.H = hbuf; q1.wts = wts; q1.status = status;
        q1.pqs = (const uint16_t*)fc1_pre_quant_scale;
        q1.act = gated ? 0 : activation;
        const int64_t fc1_groups = gated ? I / 64 : ceil_div(I, 128);
        constexpr int kTailMt = kTileTailRows / 8;
        // it reads nothing the FC1 tiles write, so it may run beside their last
        // wave (the tile kernel releases its dependents at once); it waits for
        // the tiles only before it ends (late mode 2)
        st = gated ? launch_moe_persist_mt<true>(kTailMt, q1, (int)fc1_groups, fc1_groups * E, 2, f16, s)
                   : launch_moe_persist_mt<false>(kTailMt, q1, (int)fc1_groups, fc1_groups * E, 2, f16, s);
        if (st != NVFP4_OK) return st;
        TcMoeParams t2 = t1;
        t2.fc1 = false; t2.act = 0; t2.half_stride = 0;
        t2.X = hbuf; t2.w = (const uint8_t*)fc2; t2.w_stride = nvfp4_repack_size(H, I);
        t2.N = H; t2.K = I; t2.Yp = yp; t2.H = nullptr;
        if ((st = launch_tc_moe(t2, s)) != NVFP4_OK) return st;
        MoeLinParams q2{};
        q2.w = (const uint8_t*)fc2; q2.w_stride = nvfp4_repack_size(H, I);
        q2.N = H; q2.K = I; q2.KB = round_up(I, kBlockK) / kBlockK;
        q2.splits = 1; q2.kbs = (int)q2.KB;
        q2.X = hbuf; q2.perm = perm; q2.topk = topk; q2.items = tails; q2.n_items = n_tails;
        q2.I = I; q2.Yp = yp; q2.wts = wts; q2.status = status;
        q2.early = 1;          // the routing tables are complete several launches back
        const unsigned fc2_groups = (unsigned)ceil_div(H, 128);
        // H is complete before the FC2 tiles start: beside their last wave too
        st = launch_moe_persist_mt<false>(kTailMt, q2, (int)fc2_groups, fc2_groups * E, 2, f16, s);
        if (st != NVFP4_OK) return st;
    } else {
        const int64_t est_items = moe_est_items(L, n, E);
        MoeLinParams p1{};
        p1.w = (const uint8_t*)fc1; p1.w_stride = fc1_stride; p1.half_stride = half_stride;
        p1.N = fc1_rows; p1.K = H; p1.KB = round_up(H, kBlockK) / kBlockK;
        const int64_t fc1_groups = gated ? I / 64 : ceil_div(I, 128);     // CTAs per item along the rows
        const bool persist = moe_use_persist(fc1_groups, est_items);
        p1.splits = persist ? 1 : moe_splits(fc1_groups * est_items, p1.KB, 4);
        p1.kbs = (int)ceil_div(p1.KB, p1.splits);
        p1.splits = (int)ceil_div(p1.KB, p1.kbs);
        p1.X = (const uint16_t*)X; p1.perm = perm; p1.topk = topk; p1.items = items; p1.n_items = n_items;
        p1.I = I; p1.H = hbuf; p1.wts = wts; p1.status = status;
        p1.pqs = (const uint16_t*)fc1_pre_quant_scale;
        p1.act = gated ? 0 : activation;
        const int64_t fc1_max_units = fc1_groups * L.max_items;
        if (persist)
            st = gated ? launch_moe_persist_mt<true>(L.mt, p1, (int)fc1_groups, fc1_max_units, false, f16, s)
                       : launch_moe_persist_mt<false>(L.mt, p1, (int)fc1_groups, fc1_max_units, false, f16, s);
        else
            st = gated ? launch_moe_linear_mt<true>(L.mt, p1, (unsigned)fc1_groups, (unsigned)L.max_items, f16, s)
                       : launch_moe_linear_mt<false>(L.mt, p1, (unsigned)fc1_groups, (unsigned)L.max_items, f16, s);
        if (st != NVFP4_OK) return st;

        MoeLinParams p2{};
        p2.w = (const uint8_t*)fc2; p2.w_stride = nvfp4_repack_size(H, I);
        p2.N = H; p2.K = I; p2.KB = round_up(I, kBlockK) / kBlockK;
        p2.splits = persist ? 1 : moe_splits(ceil_div(H, 128) * est_items, p2.KB, 4);
        p2.kbs = (int)ceil_div(p2.KB, p2.splits);
        p2.splits = (int)ceil_div(p2.KB, p2.kbs);
        p2.X = hbuf; p2.perm = perm; p2.topk = topk; p2.items = items; p2.n_items = n_items;
        p2.I = I; p2.Yp = yp; p2.wts = wts; p2.status = status;
        p2.early = 1;          // FC1 released it after its own wait: routing is complete
        // the routing tables were written two launches back: the persistent FC2
        // streams its first weights before waiting for FC1
        const unsigned fc2_groups = (unsigned)ceil_div(H, 128);
        st = persist ? launch_moe_persist_mt<false>(L.mt, p2, (int)fc2_groups, fc2_groups * L.max_items, true, f16, s)
                     : launch_moe_linear_mt<false>(L.mt, p2, fc2_groups, (unsigned)L.max_items, f16, s);
        if (st != NVFP4_OK) return st;
    }

    return launch_chained(f16 ? combine_kernel<true> : combine_kernel<false>,
                          dim3((unsigned)ceil_div(T * H / 4, 256)), dim3(256), 0, s,
                          "MoE combine: launch", (const float*)yp, T, topk, H, (uint16_t*)out);
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_w4a16_moe_grouped(const void* X, const float* router_logits,
                                                const void* fc1, const void* fc2,
                                                const void* fc1_pre_quant_scale,
                                                int64_t T, int E, int topk, int64_t H, int64_t I,
                                                void* out, int32_t* topk_idx_out, float* topk_weight_out,
                                                int32_t* perm_out, int32_t* offsets_out,
                                                void* workspace, size_t workspace_bytes, void* stream) {
    return moe_impl(X, router_logits, fc1, fc2, fc1_pre_quant_scale, T, E, topk, H, I, NVFP4_MOE_SWIGLU, 0, out,
                    topk_idx_out, topk_weight_out, perm_out, offsets_out, workspace, workspace_bytes, false, stream);
}

extern "C" nvfp4_status nvfp4_w4a16_moe_grouped_f16(const void* X, const float* router_logits,
                                                    const void* fc1, const void* fc2,
                                                    const void* fc1_pre_quant_scale,
                                                    int64_t T, int E, int topk, int64_t H, int64_t I,
                                                    void* out, int32_t* topk_idx_out, float* topk_weight_out,
                                                    int32_t* perm_out, int32_t* offsets_out,
                                                    void* workspace, size_t workspace_bytes, void* stream) {
    return moe_impl(X, router_logits, fc1, fc2, fc1_pre_quant_scale, T, E, topk, H, I, NVFP4_MOE_SWIGLU, 0, out,
                    topk_idx_out, topk_weight_out, perm_out, offsets_out, workspace, workspace_bytes, true, stream);
}

extern "C" nvfp4_status nvfp4_w4a16_moe_grouped_ex(const void* X, const float* router_logits,
                                                   const void* fc1, const void* fc2,
                                                   const void* fc1_pre_quant_scale,
                                                   int64_t T, int E, int topk, int64_t H, int64_t I,
                                                   int activation, int fc1_split, int f16,
                                                   void* out, int32_t* topk_idx_out, float* topk_weight_out,
                                                   int32_t* perm_out, int32_t* offsets_out,
                                                   void* workspace, size_t workspace_bytes, void* stream) {
    if (f16 != 0 && f16 != 1) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_w4a16_moe_grouped_ex: f16=%d must be 0 or 1", f16);
    return moe_impl(X, router_logits, fc1, fc2, fc1_pre_quant_scale, T, E, topk, H, I, activation, fc1_split, out,
                    topk_idx_out, topk_weight_out, perm_out, offsets_out, workspace, workspace_bytes, f16 != 0, stream);
}

// ------------------------------------------- AWQ pre-quant scale finalization --
namespace nvfp4 {
namespace {

// s[k] = max over experts of max(w3_e[k], w1_e[k]); the result is one of the
// inputs, so it converts back to the 16-bit type exactly.
template <bool F16>
__global__ void finalize_pqs_kernel(const uint16_t* __restrict__ w1, const uint16_t* __restrict__ w3, int E,
                                    int64_t H, uint16_t* __restrict__ out) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= H) return;
    auto val = [](uint16_t b) { return F16 ? f16_bits_to_f32(b) : __uint_as_float((uint32_t)b << 16); };
    float m = fmaxf(val(w1[k]), val(w3[k]));
    for (int e = 1; e < E; ++e) m = fmaxf(m, fmaxf(val(w1[(int64_t)e * H + k]), val(w3[(int64_t)e * H + k])));
    out[k] = f32_to_act_bits<F16>(m);
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_moe_finalize_pre_quant_scale(const void* w1_pre_quant_scale,
                                                           const void* w3_pre_quant_scale, int E, int64_t H,
                                                           int f16, void* out, void* stream) {
    const char* fn = "nvfp4_moe_finalize_pre_quant_scale";
    if (E < 1 || H <= 0) return fail(NVFP4_ERR_INVALID_ARG, "%s: E=%d H=%lld must be positive", fn, E, (long long)H);
    if (f16 != 0 && f16 != 1) return fail(NVFP4_ERR_INVALID_ARG, "%s: f16=%d must be 0 or 1", fn, f16);
    if (!w1_pre_quant_scale || !w3_pre_quant_scale || !out) return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(w1_pre_quant_scale, 2) || !aligned(w3_pre_quant_scale, 2) || !aligned(out, 2))
        return fail(NVFP4_ERR_ALIGNMENT, "%s: pointers must be 2-byte aligned", fn);
    const unsigned grid = (unsigned)ceil_div(H, 256);
    if (f16)
        finalize_pqs_kernel<true><<<grid, 256, 0, (cudaStream_t)stream>>>(
            (const uint16_t*)w1_pre_quant_scale, (const uint16_t*)w3_pre_quant_scale, E, H, (uint16_t*)out);
    else
        finalize_pqs_kernel<false><<<grid, 256, 0, (cudaStream_t)stream>>>(
            (const uint16_t*)w1_pre_quant_scale, (const uint16_t*)w3_pre_quant_scale, E, H, (uint16_t*)out);
    return check_cuda(cudaGetLastError(), "nvfp4_moe_finalize_pre_quant_scale: launch");
}

// ---------------------------------------------------------- dense MLP --
// The gated MLP of a dense layer: h = RN(silu(g) * u) with [g; u] = FC1(x'),
// out = RN(FC2(h)).  FC1 runs on the MoE FC1 kernels (SwiGLU fused into their
// epilogue) with one expert and the token rows as the work items; FC2 is the
// dense GEMM.
namespace nvfp4 {
namespace {

struct MlpLayout {
    size_t h, xs, gemm, total;
};

MlpLayout mlp_layout(int64_t T, int64_t H, int64_t I) {
    MlpLayout L{};
    L.h = 0;
    L.xs = (size_t)round_up(T * I * 2, 256);
    L.gemm = L.xs + (size_t)round_up(T * H * 2, 256);
    L.total = L.gemm + (size_t)round_up((int64_t)nvfp4_w4a16_gemm_workspace(T, H, I, 0), 256);
    return L;
}

// FC1 on the tile kernel when the dense shape rule picks tiles for [T, 2I]
// and the gate/up halves are whole 128-row tiles; else the streaming kernel.
bool mlp_fc1_tile(int64_t T, int64_t I) { return I % 128 == 0 && tc_tiles_fill(T, 2 * I); }

nvfp4_status mlp_impl(const void* X, const void* fc1, const void* fc2, const void* fc1_pre_quant_scale, int64_t T,
                      int64_t H, int64_t I, void* out, void* workspace, size_t workspace_bytes, bool f16,
                      void* stream) {
    const char* fn = f16 ? "nvfp4_w4a16_mlp_f16" : "nvfp4_w4a16_mlp";
    if (T < 0) return fail(NVFP4_ERR_INVALID_ARG, "%s: T=%lld is negative", fn, (long long)T);
    if (H <= 0 || I <= 0 || H % 64 != 0 || I % 64 != 0)
        return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: H=%lld and I=%lld must be positive multiples of 64", fn,
                    (long long)H, (long long)I);
    if (T == 0) return NVFP4_OK;                  // a zero-token chunk launches no kernel
    if (!X || !fc1 || !fc2 || !out) return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(X, 16) || !aligned(out, 16)) return fail(NVFP4_ERR_ALIGNMENT, "%s: X and out must be 16-byte aligned", fn);
    if (!aligned(fc1, 256) || !aligned(fc2, 256)) return fail(NVFP4_ERR_ALIGNMENT, "%s: weights must be 256-byte aligned", fn);
    if (fc1_pre_quant_scale && !aligned(fc1_pre_quant_scale, 16))
        return fail(NVFP4_ERR_ALIGNMENT, "%s: fc1_pre_quant_scale must be 16-byte aligned", fn);
    const MlpLayout L = mlp_layout(T, H, I);
    if (!workspace || workspace_bytes < L.total)
        return fail(NVFP4_ERR_WORKSPACE, "%s: workspace %zu bytes, needs %zu", fn, workspace_bytes, L.total);
    if (!aligned(workspace, 256)) return fail(NVFP4_ERR_ALIGNMENT, "%s: workspace must be 256-byte aligned", fn);
    int* status = device_status_ptr();
    if (!status) return fail(NVFP4_ERR_CUDA, "%s: no CUDA device", fn);
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* ws = (uint8_t*)workspace;
    uint16_t* hbuf = (uint16_t*)(ws + L.h);
    nvfp4_status st;

    const uint16_t* xin = (const uint16_t*)X;
    const bool fc1_tile = mlp_fc1_tile(T, I);
    if (fc1_pre_quant_scale && fc1_tile) {
        // the tile FC1 reads X through TMA: scale it into the workspace first
        // (scaling the tiles in the kernel measured slower: it doubles the
        // shared-memory traffic of a kernel bound by its shared-memory pipe)
        st = launch_awq_scale((const uint16_t*)X, (const uint16_t*)fc1_pre_quant_scale, (uint16_t*)(ws + L.xs), T, H,
                              f16, s);
        if (st != NVFP4_OK) return st;
        xin = (const uint16_t*)(ws + L.xs);
    }
    if (fc1_tile) {
        TcMoeParams t1{};
        t1.fc1 = true; t1.f16 = f16; t1.subm = T > 128 ? 2 : 1;
        t1.X = xin; t1.x_rows = T; t1.w = (const uint8_t*)fc1; t1.w_stride = 0;
        t1.N = 2 * I; t1.K = H; t1.I = I;
        t1.items = nullptr; t1.n_items = nullptr; t1.max_items = ceil_div(T, 128 * t1.subm); t1.rows = T;
        t1.H = hbuf; t1.status = status;
        if ((st = launch_tc_moe(t1, s)) != NVFP4_OK) return st;
    } else {
        const int mt = T > 8 ? 2 : 1;
        const int64_t items = ceil_div(T, 8 * mt);
        if (items > 65535) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: T=%lld too large for one call", fn, (long long)T);
        MoeLinParams p1{};
        p1.w = (const uint8_t*)fc1; p1.w_stride = 0;
        p1.N = 2 * I; p1.K = H; p1.KB = round_up(H, kBlockK) / kBlockK;
        p1.splits = moe_splits((I / 64) * items, p1.KB, 4);
        p1.kbs = (int)ceil_div(p1.KB, p1.splits);
        p1.splits = (int)ceil_div(p1.KB, p1.kbs);
        p1.X = xin; p1.perm = nullptr; p1.topk = 1; p1.items = nullptr; p1.n_items = nullptr; p1.rows = T;
        p1.I = I; p1.H = hbuf; p1.wts = nullptr; p1.status = status;
        p1.pqs = (const uint16_t*)fc1_pre_quant_scale;         // fused into the FC1 fragments
        st = mt == 1 ? launch_moe_linear<1, true>(p1, (unsigned)(I / 64), (unsigned)items, f16, s)
                     : launch_moe_linear<2, true>(p1, (unsigned)(I / 64), (unsigned)items, f16, s);
        if (st != NVFP4_OK) return st;
    }
    return run_dense_gemm(hbuf, fc2, nullptr, T, H, I, out, ws + L.gemm, workspace_bytes - L.gemm, f16, stream);
}

}  // namespace
}  // namespace nvfp4

extern "C" size_t nvfp4_w4a16_mlp_workspace(int64_t T, int64_t H, int64_t I) {
    if (T <= 0 || H <= 0 || I <= 0) return 0;
    return nvfp4::mlp_layout(T, H, I).total;
}

extern "C" nvfp4_status nvfp4_w4a16_mlp(const void* X, const void* fc1, const void* fc2,
                                        const void* fc1_pre_quant_scale, int64_t T, int64_t H, int64_t I,
                                        void* out, void* workspace, size_t workspace_bytes, void* stream) {
    return nvfp4::mlp_impl(X, fc1, fc2, fc1_pre_quant_scale, T, H, I, out, workspace, workspace_bytes, false, stream);
}

extern "C" nvfp4_status nvfp4_w4a16_mlp_f16(const void* X, const void* fc1, const void* fc2,
                                            const void* fc1_pre_quant_scale, int64_t T, int64_t H, int64_t I,
                                            void* out, void* workspace, size_t workspace_bytes, void* stream) {
    return nvfp4::mlp_impl(X, fc1, fc2, fc1_pre_quant_scale, T, H, I, out, workspace, workspace_bytes, true, stream);
}

// ------------------------------------------------- allocation-free variant --
// For callers that cannot allocate device memory themselves -- for example a
// plugin whose host framework hands it no workspace, or code that runs while
// an allocator is locked during graph construction -- this entry point runs
// the same layer on a fixed scratch area that lives in the library's own
// device memory.
namespace nvfp4 {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;     // 16 MiB
__device__ __align__(256) uint8_t g_moe_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxScratchDevices = 64;
uint8_t* g_noalloc_ptr[kMaxScratchDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
nvfp4_status noalloc_scratch(uint8_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return check_cuda(e, "nvfp4_w4a16_moe_grouped_noalloc: current device");
    if (dev < 0 || dev >= kMaxScratchDevices)
        return fail(NVFP4_ERR_CUDA, "nvfp4_w4a16_moe_grouped_noalloc: device %d not supported", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_moe_noalloc_scratch);
        if (e != cudaSuccess) return check_cuda(e, "nvfp4_w4a16_moe_grouped_noalloc: scratch address");
        g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

extern "C" size_t nvfp4_w4a16_moe_noalloc_scratch_bytes(void) { return nvfp4::kNoAllocScratchBytes; }

extern "C" nvfp4_status nvfp4_w4a16_moe_grouped_noalloc(const void* X, const float* router_logits,
                                                        const void* fc1, const void* fc2,
                                                        const void* fc1_pre_quant_scale,
                                                        int64_t T, int E, int topk, int64_t H, int64_t I,
                                                        void* out, int32_t* topk_idx_out, float* topk_weight_out,
                                                        int32_t* perm_out, int32_t* offsets_out, void* stream) {
    const size_t need = nvfp4_w4a16_moe_workspace(T, E, topk, H, I);
    if (need > nvfp4::kNoAllocScratchBytes)
        return nvfp4::fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                           "nvfp4_w4a16_moe_grouped_noalloc: T=%lld E=%d topk=%d H=%lld I=%lld needs %zu bytes "
                           "of scratch, more than the built-in %zu; use nvfp4_w4a16_moe_grouped with a workspace",
                           (long long)T, E, topk, (long long)H, (long long)I, need, nvfp4::kNoAllocScratchBytes);
    if (T <= 0 || need == 0)    // nothing to run, or arguments the regular entry point rejects
        return nvfp4_w4a16_moe_grouped(X, router_logits, fc1, fc2, fc1_pre_quant_scale, T, E, topk, H, I, out,
                                       topk_idx_out, topk_weight_out, perm_out, offsets_out, nullptr, 0, stream);
    uint8_t* scratch = nullptr;
    const nvfp4_status st = nvfp4::noalloc_scratch(&scratch);
    if (st != NVFP4_OK) return st;
    return nvfp4_w4a16_moe_grouped(X, router_logits, fc1, fc2, fc1_pre_quant_scale, T, E, topk, H, I, out,
                                   topk_idx_out, topk_weight_out, perm_out, offsets_out, scratch,
                                   nvfp4::kNoAllocScratchBytes, stream);
}
