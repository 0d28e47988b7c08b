/*
 * nvfp4_w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 NVFP4 weight-only GEMM library.
 *
 * The method: weights are NVFP4 -- 4-bit E2M1 codes (sign bit + magnitudes
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}), one float8_e4m3fn scale per 16 consecutive K
 * elements, one FP32 global scale per tensor -- and activations stay 16-bit
 * (BF16, or FP16 through the *_f16 entry points); the activation is never
 * quantized.  Every forward step computes, with RN the round-to-nearest-even
 * conversion to the activation type,
 *     W[n,k] = RN( e2m1(code[n,k]) * e4m3(scale[n,k/16]) * g )
 *     Y[m,n] = RN( sum_k x'[m,k] * W[n,k] )            (FP32 accumulation)
 * with x' = x, or x' = RN(x * pre_quant_scale) for AWQ checkpoints.
 * Sources: "[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt on Hopper"
 * (TensorRT-LLM PR 14775), Description and Changes table (on-the-fly NVFP4
 * dequant: E2M1 codebook lookup, per-block FP8 scale, per-tensor scale;
 * active-expert-only MoE dequant; CUDA-graph capturable); SGLang PR 40022,
 * Motivation and Modifications (gs=16, E4M3 group scales, a real global scale
 * stored as a divisor that must be inverted); "[None][fix] Apply the NVFP4_AWQ
 * pre-quant scale in MegaMoE CuteDSL" (TensorRT-LLM PR 20823), Description
 * (x * pre_quant_scale in BF16 before the GEMM, shape [1, hidden]; a zero-token
 * chunk launches no kernel; an already-quantized activation is refused);
 * "[TRTLLM-12720][feat] Support nvfp4 w4a16 on sm120" (TensorRT-LLM PR 16511),
 * Summary (W4A16 = FP4 weights with BF16 or FP16 activations).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers on the current CUDA device unless
 *    stated otherwise; all calls are asynchronous on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream).  The library never allocates, frees or
 *    synchronizes (except nvfp4_device_status, which synchronizes `stream`).
 *  - The caller owns every buffer.  BF16 and FP16 tensors are passed as raw
 *    16-bit patterns (uint16_t / void*), row-major, densely packed.
 *  - Arguments are validated before anything is launched; a failed check
 *    returns a non-OK status, launches nothing and sets a message readable
 *    with nvfp4_last_error() (thread-local).
 *  - No call reads device memory back to the host, so every GEMM / MoE /
 *    dequant call can be captured in a CUDA graph.
 *  - Faults inside a kernel that the host cannot see (a repacked-weight header
 *    whose magic or shape does not match the call, a pipeline wait that ran
 *    out of its iteration limit) do not trap: the kernel skips its work and
 *    records an error code in a per-device status word, which
 *    nvfp4_device_status() returns.
 */
#ifndef NVFP4_W4A16_H
#define NVFP4_W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad flag, non-finite divisor */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 2, /* K not a positive multiple of 16, sizes beyond the limits */
    NVFP4_ERR_ALIGNMENT = 3,         /* a pointer not aligned as documented */
    NVFP4_ERR_WORKSPACE = 4,         /* workspace missing or smaller than the query says */
    NVFP4_ERR_CUDA = 5,              /* a CUDA runtime call failed (message has the CUDA error) */
    NVFP4_ERR_TIMEOUT = 6,           /* device status: a pipeline wait exceeded its limit */
    NVFP4_ERR_BAD_WEIGHT = 7         /* device status: repacked header magic/shape mismatch */
} nvfp4_status;

/* Version of this ABI (bumped on any incompatible change). */
int nvfp4_abi_version(void);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* nvfp4_last_error(void);

/*
 * Per-device status word written by kernels (0 = OK, else an nvfp4_status).
 * Synchronizes `stream`, copies the word of the current device to *code_out
 * and, if `clear` != 0, resets it to 0.
 */
nvfp4_status nvfp4_device_status(int* code_out, int clear, void* stream);

/* ------------------------------------------------------------------------ */
/* Repack (once per weight tensor, at load time)                             */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of the repacked form of an N x K NVFP4 weight (0 if N <= 0, or K is
 * not a positive multiple of 16).  The size is a multiple of 256.
 */
size_t nvfp4_repack_size(int64_t N, int64_t K);

/*
 * Rewrite a checkpoint-layout NVFP4 weight into the library's tiled layout.
 * This is the "load" step (the pages' Marlin repack / derived-buffer refresh):
 * a pure function of its inputs, so re-running it gives identical bytes.
 *
 *  packed       device, uint8 [N, K/2] row-major; byte (n, j) holds code (n, 2j)
 *               in its low nibble and code (n, 2j+1) in its high nibble.
 *  scales_e4m3  device, uint8 [N, K/16] row-major float8_e4m3fn codes.
 *  global_scale FP32 per-tensor global scale, by value.
 *  global_is_divisor  1: global_scale is stored as a divisor d (compressed-
 *               tensors convention) and the multiplier is g = RN_fp32(1/d),
 *               one IEEE division done on the host; 0: g = global_scale.
 *               g must be finite and nonzero.
 *  out          device, 256-byte aligned, out_bytes >= nvfp4_repack_size(N, K).
 *
 * Layout of `out` (all offsets in bytes):
 *  [0, 256)      header: u32 magic 0x34504E56, u32 version, i64 N, i64 K,
 *                i64 Np (N rounded up to 256), i64 Kp (K rounded up to 64),
 *                f32 g, f32 global_scale, u32 global_is_divisor.
 *  [256, 4352)   BF16 magnitude table: 256 entries of 16 bytes, entry s = the
 *                BF16 values RN_bf16(mag_j * e4m3(s) * g) of the 8 E2M1
 *                magnitudes j = 0..7, stored as 8 low bytes then 8 high bytes.
 *  [4352, 8448)  FP16 magnitude table: the same with RN_f16 (IEEE binary16;
 *                products beyond 65504 round to infinity).
 *  [8448, ...)   atoms of 16 rows x 64 k (576 bytes each), ordered by
 *                256-row tile, then 64-k block, then 16-row block.  In an atom,
 *                lane L = 4r + q (r < 8, q < 4) owns 16 code bytes at 16L
 *                (rows r and r+8 of the block, k group q, 8 bytes each) and 2
 *                scale bytes at 512 + 2L.  Each 32-bit code word holds 8
 *                consecutive k: magnitude of element i in bits 4i..4i+2 and
 *                the signs of elements 0..7 in bits 7, 15, 23, 31, 3, 11, 19, 27.
 *                Rows >= N and k >= K are padded with code 0 and scale 0.
 */
nvfp4_status nvfp4_repack(const uint8_t* packed, const uint8_t* scales_e4m3,
                          float global_scale, int global_is_divisor,
                          int64_t N, int64_t K,
                          void* out, size_t out_bytes, void* stream);

/*
 * Scales in the checkpoint's swizzled layout.  The source pages keep NVFP4
 * per-block scales swizzled and derive the linear view ("[TRTLLM-12288][feat]
 * Support Nemotron-H nvfp4 ckpt on Hopper", Linear: "Per-block scales stay in
 * swizzled layout; the unswizzled view is a derived non-persistent buffer")
 * without printing the layout; the one read here is the 128 x 4 tile layout of
 * NVIDIA's block-scaled GEMMs: rows padded to 128 and 16-groups to 4, tiles of
 * 128 rows x 4 groups stored row-tile-major (512 bytes each), and inside a
 * tile the scale of row r (0..127), group c (0..3) at (r % 32)*16 + (r / 32)*4 + c.
 * nvfp4_repack_ex with scale_layout = NVFP4_SCALES_SWIZZLED_128x4 reads
 * scales_e4m3 in that layout (nvfp4_swizzled_scales_size(N, K) bytes, padding
 * ignored) and writes exactly what nvfp4_repack writes from the linear view;
 * NVFP4_SCALES_LINEAR is nvfp4_repack.
 */
typedef enum { NVFP4_SCALES_LINEAR = 0, NVFP4_SCALES_SWIZZLED_128x4 = 1 } nvfp4_scale_layout;

size_t nvfp4_swizzled_scales_size(int64_t N, int64_t K);
nvfp4_status nvfp4_repack_ex(const uint8_t* packed, const uint8_t* scales_e4m3, int scale_layout,
                             float global_scale, int global_is_divisor,
                             int64_t N, int64_t K,
                             void* out, size_t out_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Standalone dequant                                                        */
/* ------------------------------------------------------------------------ */

/*
 * W (BF16, [N, K] row-major) from a repacked weight: exactly the operand the
 * GEMM kernels feed to the tensor cores.
 *  repacked  device, as written by nvfp4_repack for the same N, K.
 *  out_bf16  device, N*K uint16, 16-byte aligned.
 */
nvfp4_status nvfp4_dequant(const void* repacked, int64_t N, int64_t K,
                           uint16_t* out_bf16, void* stream);

/* The same with FP16 output: the operand of the *_f16 GEMM entry points. */
nvfp4_status nvfp4_dequant_f16(const void* repacked, int64_t N, int64_t K,
                               uint16_t* out_f16, void* stream);

/* ------------------------------------------------------------------------ */
/* Dense W4A16 GEMM                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Workspace bytes nvfp4_w4a16_gemm needs for this problem (may be 0).
 */
size_t nvfp4_w4a16_gemm_workspace(int64_t M, int64_t N, int64_t K, int has_pre_quant_scale);

/*
 * Y = X' . W^T with X' = X (pre_quant_scale == NULL) or RN_bf16(X * pre_quant_scale).
 *  X               device BF16 [M, K] row-major, 16-byte aligned.
 *  repacked        device, from nvfp4_repack(N, K).
 *  pre_quant_scale device BF16 [K] or NULL (AWQ per-channel scale).
 *  Y               device BF16 [M, N] row-major, 4-byte aligned.
 *  workspace       device, >= nvfp4_w4a16_gemm_workspace(...) bytes, 256-byte
 *                  aligned (may be NULL when that size is 0).  Contents on entry
 *                  do not matter.
 * M == 0 or N == 0 returns NVFP4_OK and launches nothing.  M <= 16 (and, up
 * to M = 511, shapes whose output tiles would leave most SMs idle) runs the
 * split-K HBM-streaming decode kernel; other shapes one of two tensor-core
 * tile kernels (dequantized weight in shared memory, or in tensor memory as
 * the MMA's A operand), chosen per shape; results agree within rounding.
 * The decode kernel applies pre_quant_scale to the activation fragments it
 * feeds to the MMAs (one packed BF16/FP16 multiply, the same single rounding),
 * so it needs no workspace and no extra launch; the tile kernels write X' into
 * the workspace first.
 * The GEMM kernels use programmatic dependent launch: they may begin reading
 * the repacked weight before the preceding kernel of the stream has finished
 * (only if that kernel itself allows its dependents to start early), and read
 * X / write Y only after it has.  So a kernel that rewrites the repacked
 * weight must not be such an early-release kernel directly before the GEMM.
 * The tile kernels are launched in stream order but allow the kernel after
 * them to start early (it still waits for them before touching their output).
 */
nvfp4_status nvfp4_w4a16_gemm(const void* X, const void* repacked, const void* pre_quant_scale,
                              int64_t M, int64_t N, int64_t K, void* Y,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP16 activations: the same call with X, pre_quant_scale and Y in FP16, the
 * weight dequantized to FP16 and every RN an FP16 rounding (results beyond
 * 65504 in magnitude become infinities).  Same kernels, FP16 tensor-core
 * MMAs, same workspace size.
 */
nvfp4_status nvfp4_w4a16_gemm_f16(const void* X, const void* repacked, const void* pre_quant_scale,
                                  int64_t M, int64_t N, int64_t K, void* Y,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * The launch plan nvfp4_w4a16_gemm / _f16 use for an M x N x K problem on the
 * current device (the SM count decides wave sizes; without a device 148 SMs
 * are assumed).  Host only: nothing is launched, no device memory is touched.
 *  has_pre_quant_scale  0 or 1 (an AWQ scale adds one activation pass).
 *  kernel_out    -1 nothing (M or N is 0), 0 split-K streaming decode kernel,
 *                1 tile kernel with the dequantized weight in shared memory,
 *                2 tile kernel with the dequantized weight in tensor memory.
 *  tokens_out    activation rows per CTA tile (8 or 16 in the decode kernel).
 *  splits_out    K splits (the decode kernel sums them inside a thread-block
 *                cluster; the tile kernels add one FP32 reduction pass).
 *  launches_out  kernels one call launches.
 * Errors as nvfp4_w4a16_gemm's argument checks (null output pointer,
 * negative size, K not a positive multiple of 16).
 */
nvfp4_status nvfp4_w4a16_gemm_plan(int64_t M, int64_t N, int64_t K, int has_pre_quant_scale,
                                   int* kernel_out, int* tokens_out, int* splits_out, int* launches_out);

/* ------------------------------------------------------------------------ */
/* Grouped top-k MoE layer (FC1 gate/up + SwiGLU, FC2, weighted combine)     */
/* ------------------------------------------------------------------------ */

/*
 * The MoE layer's routing step on its own (the same results as the layer's
 * own routing; the kernels are the layer's up to 512 tokens, above which the
 * layer uses chunked kernels that need its workspace while this call keeps
 * a single-CTA permutation): per token the top-k of its FP32 router logits
 * (ties to the lower expert index, slots in descending-logit order) and
 * p = softmax over the k selected logits; then the routing slots s = t*topk + j sorted by expert,
 * then token, then slot (stable).  "[TRTLLM-12288][feat] Support Nemotron-H
 * nvfp4 ckpt on Hopper", Changes table (MoE: only the routed, active experts'
 * weights are dequantized -- the permutation groups each expert's rows).
 *  router_logits    device FP32 [T, E].
 *  topk_idx_out     device int32 [T, topk]: selected experts.
 *  topk_weight_out  device FP32 [T, topk]: routing weights p.
 *  perm_out         device int32 [T*topk]: perm[i] = the slot at sorted position i.
 *  inv_out          device int32 [T*topk]: its inverse, inv[perm[i]] = i.
 *  offsets_out      device int32 [E+1]: exclusive scan of the per-expert slot
 *                   counts (expert e owns sorted positions [offsets[e], offsets[e+1])).
 * All outputs are required and 4-byte aligned.  Limits as the layer: E <= 256,
 * topk <= 16, topk <= E, T*topk < 2^31.  T == 0 returns NVFP4_OK and launches
 * nothing (no output is written).  No workspace.
 */
nvfp4_status nvfp4_moe_route(const float* router_logits, int64_t T, int E, int topk,
                             int32_t* topk_idx_out, float* topk_weight_out, int32_t* perm_out,
                             int32_t* inv_out, int32_t* offsets_out, void* stream);

size_t nvfp4_w4a16_moe_workspace(int64_t T, int E, int topk, int64_t H, int64_t I);

/*
 * out[t] = RN_bf16( sum_j p[t,j] * FC2_e( RN_bf16( silu(g) * u ) ) ), e = idx[t,j],
 * [g; u] = FC1_e(x'_t), for the top-k experts of each token.
 *  X                 device BF16 [T, H].
 *  router_logits     device FP32 [T, E].  Top-k on the logits, ties to the lower
 *                    expert index, slots in descending-logit order; p = softmax
 *                    over the k selected logits.
 *  fc1               device: E repacked [2I, H] weights back to back, expert e at
 *                    fc1 + e * nvfp4_repack_size(2I, H); rows [0, I) are the gate
 *                    projection, rows [I, 2I) the up projection.
 *  fc2               device: E repacked [H, I] weights, expert e at
 *                    fc2 + e * nvfp4_repack_size(H, I).
 *  fc1_pre_quant_scale  device BF16 [H] or NULL (AWQ scale on FC1's input).
 *  out               device BF16 [T, H].
 *  topk_idx_out      device int32 [T, topk] or NULL; topk_weight_out FP32 [T, topk]
 *                    or NULL; perm_out int32 [T*topk] or NULL (routing slots t*topk+j
 *                    sorted by expert, then token, then slot); offsets_out int32
 *                    [E+1] or NULL (exclusive scan of per-expert counts).
 * Only the weights of experts that received at least one token are read.
 * T == 0 returns NVFP4_OK and launches nothing.  Limits: E <= 256, topk <= 16,
 * topk <= E, H and I multiples of 64, T * topk / 8 + E below 65536 (one call).
 * workspace: >= nvfp4_w4a16_moe_workspace(...) bytes, 256-byte aligned; it holds
 * the routing tables, the intermediate activations and the FP32 per-slot rows.
 */
nvfp4_status nvfp4_w4a16_moe_grouped(const void* X, const float* router_logits,
                                     const void* fc1, const void* fc2,
                                     const void* fc1_pre_quant_scale,
                                     int64_t T, int E, int topk, int64_t H, int64_t I,
                                     void* out, int32_t* topk_idx_out, float* topk_weight_out,
                                     int32_t* perm_out, int32_t* offsets_out,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP16 activations: X, fc1_pre_quant_scale and out in FP16; the expert weights,
 * h and out rounded to FP16.  Routing is unchanged (FP32 logits).
 */
nvfp4_status nvfp4_w4a16_moe_grouped_f16(const void* X, const float* router_logits,
                                         const void* fc1, const void* fc2,
                                         const void* fc1_pre_quant_scale,
                                         int64_t T, int E, int topk, int64_t H, int64_t I,
                                         void* out, int32_t* topk_idx_out, float* topk_weight_out,
                                         int32_t* perm_out, int32_t* offsets_out,
                                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * MoE layer variants.  activation: the expert type -- NVFP4_MOE_SWIGLU (gated:
 * h = RN(silu(g) * u), the default of nvfp4_w4a16_moe_grouped), NVFP4_MOE_RELU2
 * (non-gated: h = RN(max(v, 0)^2)) or NVFP4_MOE_SILU (non-gated: h =
 * RN(silu(v))), v = FC1_e(x'); non-gated experts have fc1 = E repacked [I, H]
 * weights, expert e at fc1 + e * nvfp4_repack_size(I, H) (SGLang PR 40022,
 * review thread: relu2 and silu non-gated experts).  fc1_split = 1 (gated
 * only): the gate and up projections were quantized separately, each with its
 * own global scale (per-shard w1/w3 globals, same thread), and are repacked
 * separately as two [I, H] weights: expert e's gate at fc1 + e * 2 * S and its
 * up projection at fc1 + (2e + 1) * S, S = nvfp4_repack_size(I, H).  f16 = 1
 * for FP16 activations.  Everything else as nvfp4_w4a16_moe_grouped; the
 * workspace size is the same.
 */
typedef enum { NVFP4_MOE_SWIGLU = 0, NVFP4_MOE_RELU2 = 1, NVFP4_MOE_SILU = 2 } nvfp4_moe_activation;

nvfp4_status nvfp4_w4a16_moe_grouped_ex(const void* X, const float* router_logits,
                                        const void* fc1, const void* fc2,
                                        const void* fc1_pre_quant_scale,
                                        int64_t T, int E, int topk, int64_t H, int64_t I,
                                        int activation, int fc1_split, int f16,
                                        void* out, int32_t* topk_idx_out, float* topk_weight_out,
                                        int32_t* perm_out, int32_t* offsets_out,
                                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * The kernels nvfp4_w4a16_moe_grouped* would run for a problem on the current
 * device (host only, no launch).  activation as nvfp4_w4a16_moe_grouped_ex.
 *  path_out           0 nothing (T == 0); 1 streaming kernels, one CTA per
 *                     (work item, column group) with K split across a thread-
 *                     block cluster; 2 streaming kernels, one persistent wave
 *                     that walks the (work item, column group) units with K
 *                     whole; 3 gathered rows on the tcgen05 tile kernels;
 *                     4 one token with topk <= 8: two kernels in all (every
 *                     CTA routes the token itself; FC2 sums the slots'
 *                     weighted outputs inside a cluster, so no routing or
 *                     combine kernel runs).
 *  rows_per_item_out  routed rows per work item (8 or 16 streaming, 128 or
 *                     256 on the tile kernels; 0 when T == 0).
 * The choice depends on the routed rows per expert on average (T * topk / E)
 * and, on the streaming path, on the expected units per SM.  Errors as the
 * layer's argument checks (null output pointer, sizes outside its limits).
 */
nvfp4_status nvfp4_w4a16_moe_plan(int64_t T, int E, int topk, int64_t H, int64_t I, int activation,
                                  int* path_out, int* rows_per_item_out);

/*
 * The layer's FC1 activation scale from per-expert AWQ pre-quant scales (a
 * load-time step): out[k] = max over experts e of max(w3_e[k], w1_e[k])
 * ("[None][fix] Apply the NVFP4_AWQ pre-quant scale in MegaMoE CuteDSL",
 * Description: the finalization writes max(w3, w1) into the [1, hidden] FC1
 * input scale).  w1_pre_quant_scale, w3_pre_quant_scale: device [E, H] BF16
 * (FP16 when f16 = 1); out: device [H], the fc1_pre_quant_scale of the MoE
 * calls.  NaN entries are ignored by the max.
 */
nvfp4_status nvfp4_moe_finalize_pre_quant_scale(const void* w1_pre_quant_scale,
                                                const void* w3_pre_quant_scale, int E, int64_t H,
                                                int f16, void* out, void* stream);

/* ------------------------------------------------------------------------ */
/* Dense gated MLP (FC1 gate/up + SwiGLU, FC2)                               */
/* ------------------------------------------------------------------------ */

size_t nvfp4_w4a16_mlp_workspace(int64_t T, int64_t H, int64_t I);

/*
 * out[t] = RN( FC2( RN( silu(g) * u ) ) ), [g; u] = FC1(x'_t): the MoE layer's
 * expert computation on one dense weight pair, for every token (the SwiGLU of
 * gated experts: SGLang PR 40022, review thread on is_gated; the fused gate/up
 * FC1 "w3_w1" of "[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt on Hopper",
 * Changes table).  RN rounds to BF16 (or FP16 for the _f16 entry point).
 *  X                  device [T, H], 16-byte aligned.
 *  fc1                device, repacked [2I, H]: rows [0, I) gate, [I, 2I) up.
 *  fc2                device, repacked [H, I].
 *  fc1_pre_quant_scale device [H] or NULL (AWQ scale on FC1's input).
 *  out                device [T, H], 16-byte aligned.
 *  workspace          >= nvfp4_w4a16_mlp_workspace(T, H, I) bytes, 256-byte
 *                     aligned; holds h [T, I] and the scaled activation.
 * H and I positive multiples of 64; T == 0 returns NVFP4_OK and launches nothing.
 * FC1 runs the MoE FC1 kernels (SwiGLU fused into the epilogue, h never in
 * FP32 memory), FC2 the dense GEMM.
 */
nvfp4_status nvfp4_w4a16_mlp(const void* X, const void* fc1, const void* fc2,
                             const void* fc1_pre_quant_scale, int64_t T, int64_t H, int64_t I,
                             void* out, void* workspace, size_t workspace_bytes, void* stream);
nvfp4_status nvfp4_w4a16_mlp_f16(const void* X, const void* fc1, const void* fc2,
                                 const void* fc1_pre_quant_scale, int64_t T, int64_t H, int64_t I,
                                 void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free variant of nvfp4_w4a16_moe_grouped (no counterpart in the
 * source pages: it exists for callers that cannot allocate device memory, such
 * as a plugin whose host framework gives it no workspace, or code running
 * while allocation is not allowed).  Same arguments and results, minus the
 * workspace: the layer runs on a scratch array of
 * nvfp4_w4a16_moe_noalloc_scratch_bytes() bytes (16 MiB) that is a static
 * device variable of this library, so every GPU that loads the library holds
 * it until the process exits.  Problems whose nvfp4_w4a16_moe_workspace()
 * exceeds that size are rejected with NVFP4_ERR_UNSUPPORTED_SHAPE (with
 * E=128, topk=8, H=2048, I=768 that allows up to T=215 tokens per call).  The entry point itself calls
 * no allocating routine.  The first call on a device looks the scratch address
 * up (cudaGetSymbolAddress, which may load the library's device code), so make
 * that first call before any stream capture.  Every call shares the one array;
 * nothing in it has to start at zero, but calls that overlap on the GPU (on
 * different streams) race on it and give wrong results.  The looked-up address
 * (like that of the status word behind nvfp4_device_status) is kept for the
 * life of the process, so the library must not be used across a reset of the
 * device (cudaDeviceReset), which may load its device code at another address.
 */
size_t nvfp4_w4a16_moe_noalloc_scratch_bytes(void);
nvfp4_status nvfp4_w4a16_moe_grouped_noalloc(const void* X, const float* router_logits,
                                             const void* fc1, const void* fc2,
                                             const void* fc1_pre_quant_scale,
                                             int64_t T, int E, int topk, int64_t H, int64_t I,
                                             void* out, int32_t* topk_idx_out, float* topk_weight_out,
                                             int32_t* perm_out, int32_t* offsets_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_W4A16_H */
