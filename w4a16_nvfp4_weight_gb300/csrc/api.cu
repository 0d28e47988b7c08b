// Host side of the C ABI: error reporting, the device status word, and the
// dense GEMM entry point (argument validation and the decode / tile shape rule).
//
// Boundary behaviour follows the pages: validate shapes, strides and scales
// with descriptive errors before launching ("[TRTLLM-12288][feat] Support
// Nemotron-H nvfp4 ckpt on Hopper", review of the dequant wrappers and of the
// FP8-input guard: fail fast instead of reading wrong addresses), keep the call
// capturable in a CUDA graph (same page, Description), and refuse anything but
// BF16 activations ("[None][fix] Apply the NVFP4_AWQ pre-quant scale in MegaMoE
// CuteDSL": already-quantized inputs are rejected).
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "gemm_decode.cuh"
#include "gemm_tc.cuh"

namespace nvfp4 {

namespace {
thread_local char g_msg[512] = "";
__device__ int g_status_word;
constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::mutex g_mu;
}  // namespace

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
}

nvfp4_status fail(nvfp4_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

nvfp4_status check_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return NVFP4_OK;
    return fail(NVFP4_ERR_CUDA, "%s: CUDA error %d (%s)", what, (int)e, cudaGetErrorString(e));
}

int* device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_status_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

// Split-K plan of the decode kernel for an M x N x K problem.
struct DecodePlan {
    int MT, ring, W, splits, kbs;
    int64_t ctas;
    bool ok;
};

DecodePlan plan_decode(int64_t M, int64_t N, int64_t K, bool f16, bool awq) {
    const int MT = M <= 8 ? 1 : 2;
    const int64_t TOK = 8 * MT;
    const int64_t KB = round_up(K, kBlockK) / kBlockK;
    const int64_t mchunks = ceil_div(M, TOK);
    const int64_t sms = sm_count();
    // Split K until the CTAs fill one wave (as many per SM as shared memory
    // holds), with at most 8 CTAs per cluster (larger, non-portable clusters
    // measured slower) and at least two 64-k blocks per CTA.
    auto plan_for = [&](int ring, int W) {
        DecodePlan pl{};
        pl.MT = MT; pl.ring = ring; pl.W = W; pl.ok = true;
        const int64_t base = ceil_div(N, (int64_t)W * kAtomRows) * mchunks;
        const int64_t target = (int64_t)decode_ctas_per_sm(MT, ring, W, f16, awq) * sms;
        int64_t splits = std::max<int64_t>(1, target / std::max<int64_t>(base, 1));
        splits = std::min<int64_t>(splits, std::min<int64_t>(8, std::max<int64_t>(1, KB / 2)));
        const int64_t kbs = ceil_div(KB, splits);
        pl.splits = (int)ceil_div(KB, kbs);
        pl.kbs = (int)kbs;
        pl.ctas = base * pl.splits;
        return pl;
    };
    // Slices of at most 16 blocks spend much of their time filling the ring
    // and reducing: those take the shallow ring, which packs more CTAs per SM,
    // when that buys a finer split.
    auto plan_rings = [&](int W) {
        DecodePlan pl = plan_for(kRingDeep, W);
        if (pl.kbs <= 16) {
            const DecodePlan shallow = plan_for(kRingShallow, W);
            if (shallow.splits > pl.splits) pl = shallow;
        }
        return pl;
    };
    DecodePlan pl = plan_rings(8);
    // A grid of 128-row CTAs that fills under three quarters of a wave (few
    // output rows, the split capped by the cluster size) leaves SMs idle -- the
    // block scheduler also stacks such grids' clusters on part of the SMs --
    // so it takes 64-row CTAs instead, twice as many.
    const int64_t wave = (int64_t)decode_ctas_per_sm(MT, pl.ring, 8, f16, awq) * sms;
    if (pl.ctas * 4 < wave * 3) {
        const DecodePlan half = plan_rings(4);
        if (half.ctas > pl.ctas) pl = half;
    }
    return pl;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" int nvfp4_abi_version(void) { return 2; }

extern "C" const char* nvfp4_last_error(void) { return g_msg; }

extern "C" nvfp4_status nvfp4_device_status(int* code_out, int clear, void* stream) {
    if (!code_out) return fail(NVFP4_ERR_INVALID_ARG, "nvfp4_device_status: code_out is null");
    int* p = device_status_ptr();
    if (!p) return fail(NVFP4_ERR_CUDA, "nvfp4_device_status: status word unavailable");
    nvfp4_status st = check_cuda(cudaStreamSynchronize((cudaStream_t)stream), "nvfp4_device_status: synchronize");
    if (st != NVFP4_OK) return st;
    int v = 0;
    st = check_cuda(cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost), "nvfp4_device_status: read");
    if (st != NVFP4_OK) return st;
    if (clear) {
        st = check_cuda(cudaMemset(p, 0, sizeof(int)), "nvfp4_device_status: clear");
        if (st != NVFP4_OK) return st;
    }
    *code_out = v;
    return NVFP4_OK;
}

extern "C" size_t nvfp4_w4a16_gemm_workspace(int64_t M, int64_t N, int64_t K, int has_pre_quant_scale) {
    if (M <= 0 || N <= 0 || K <= 0 || K % kGroup != 0) return 0;
    if (use_tc_path(M, N, K)) return tc_workspace_bytes(M, N, K, has_pre_quant_scale != 0);
    return 0;               // the decode kernel applies AWQ to its activation fragments
}

nvfp4_status nvfp4::run_dense_gemm(const void* X, const void* repacked, const void* pre_quant_scale, int64_t M,
                                   int64_t N, int64_t K, void* Y, void* workspace, size_t workspace_bytes, bool f16,
                                   void* stream) {
    const char* fn = f16 ? "nvfp4_w4a16_gemm_f16" : "nvfp4_w4a16_gemm";
    if (M < 0 || N < 0) return fail(NVFP4_ERR_INVALID_ARG, "%s: negative size M=%lld N=%lld", fn, (long long)M, (long long)N);
    if (K <= 0 || K % kGroup != 0) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: K=%lld must be a positive multiple of 16", fn, (long long)K);
    if (M == 0 || N == 0) return NVFP4_OK;          // nothing to compute, nothing launched
    if (!X || !repacked || !Y) return fail(NVFP4_ERR_INVALID_ARG, "%s: null pointer (X=%p W=%p Y=%p)", fn, X, repacked, Y);
    if (!aligned(X, 16)) return fail(NVFP4_ERR_ALIGNMENT, "%s: X must be 16-byte aligned", fn);
    if (!aligned(repacked, 256)) return fail(NVFP4_ERR_ALIGNMENT, "%s: repacked weight must be 256-byte aligned", fn);
    if (!aligned(Y, 4)) return fail(NVFP4_ERR_ALIGNMENT, "%s: Y must be 4-byte aligned", fn);
    if (pre_quant_scale && !aligned(pre_quant_scale, 16)) return fail(NVFP4_ERR_ALIGNMENT, "%s: pre_quant_scale must be 16-byte aligned", fn);
    const size_t need = nvfp4_w4a16_gemm_workspace(M, N, K, pre_quant_scale != nullptr);
    if (workspace_bytes < need || (need > 0 && workspace == nullptr))
        return fail(NVFP4_ERR_WORKSPACE, "%s: workspace %zu bytes, needs %zu", fn, workspace_bytes, need);
    if (need > 0 && !aligned(workspace, 256)) return fail(NVFP4_ERR_ALIGNMENT, "%s: workspace must be 256-byte aligned", fn);
    int* status = device_status_ptr();
    if (!status) return fail(NVFP4_ERR_CUDA, "%s: no CUDA device", fn);
    cudaStream_t s = (cudaStream_t)stream;
    if (use_tc_path(M, N, K)) {
        TcParams tp{};
        tp.X = (const uint16_t*)X; tp.pqs = (const uint16_t*)pre_quant_scale;
        tp.rp = (const uint8_t*)repacked; tp.Y = (uint16_t*)Y;
        tp.M = M; tp.N = N; tp.K = K; tp.status = status; tp.f16 = f16;
        tp.workspace = workspace; tp.workspace_bytes = workspace_bytes;
        return launch_tc(tp, s);
    }
    const DecodePlan pl = plan_decode(M, N, K, f16, pre_quant_scale != nullptr);
    if (!pl.ok) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: K=%lld too large for the decode kernel", fn, (long long)K);
    DecodeParams p{};
    p.X = (const uint16_t*)X; p.pqs = (const uint16_t*)pre_quant_scale;
    p.rp = (const uint8_t*)repacked; p.Y = (uint16_t*)Y;
    p.M = M; p.N = N; p.K = K;
    p.KB = round_up(K, kBlockK) / kBlockK;
    p.kbs = pl.kbs; p.splits = pl.splits; p.status = status;
    return launch_decode(p, pl.MT, pl.ring, pl.W, f16, s);
}

extern "C" nvfp4_status nvfp4_w4a16_gemm(const void* X, const void* repacked, const void* pre_quant_scale,
                                         int64_t M, int64_t N, int64_t K, void* Y,
                                         void* workspace, size_t workspace_bytes, void* stream) {
    return run_dense_gemm(X, repacked, pre_quant_scale, M, N, K, Y, workspace, workspace_bytes, false, stream);
}

extern "C" nvfp4_status nvfp4_w4a16_gemm_plan(int64_t M, int64_t N, int64_t K, int has_pre_quant_scale,
                                              int* kernel_out, int* tokens_out, int* splits_out,
                                              int* launches_out) {
    const char* fn = "nvfp4_w4a16_gemm_plan";
    if (!kernel_out || !tokens_out || !splits_out || !launches_out)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: null output pointer", fn);
    if (M < 0 || N < 0) return fail(NVFP4_ERR_INVALID_ARG, "%s: negative size M=%lld N=%lld", fn, (long long)M, (long long)N);
    if (K <= 0 || K % kGroup != 0) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: K=%lld must be a positive multiple of 16", fn, (long long)K);
    if (has_pre_quant_scale != 0 && has_pre_quant_scale != 1)
        return fail(NVFP4_ERR_INVALID_ARG, "%s: has_pre_quant_scale=%d must be 0 or 1", fn, has_pre_quant_scale);
    if (M == 0 || N == 0) {
        *kernel_out = -1; *tokens_out = 0; *splits_out = 0; *launches_out = 0;
        return NVFP4_OK;
    }
    if (use_tc_path(M, N, K)) {
        bool wa = false;
        int tok = 0, sp = 1;
        tc_plan_info(M, N, K, &wa, &tok, &sp);
        *kernel_out = wa ? 2 : 1; *tokens_out = tok; *splits_out = sp;
        *launches_out = 1 + (sp > 1 ? 1 : 0) + has_pre_quant_scale;
        return NVFP4_OK;
    }
    const DecodePlan pl = plan_decode(M, N, K, false, has_pre_quant_scale != 0);
    if (!pl.ok) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "%s: K=%lld too large for the decode kernel", fn, (long long)K);
    *kernel_out = 0; *tokens_out = 8 * pl.MT; *splits_out = pl.splits;
    *launches_out = 1;            // AWQ is applied inside the decode kernel
    return NVFP4_OK;
}

extern "C" nvfp4_status nvfp4_w4a16_gemm_f16(const void* X, const void* repacked, const void* pre_quant_scale,
                                             int64_t M, int64_t N, int64_t K, void* Y,
                                             void* workspace, size_t workspace_bytes, void* stream) {
    return run_dense_gemm(X, repacked, pre_quant_scale, M, N, K, Y, workspace, workspace_bytes, true, stream);
}
