// api.cu -- configuration checks, workspace layout, the grouped-GEMM dispatch, the gate
// entry point and moe_forward (the whole layer on one stream).
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "gemm.h"
#include "sm100.cuh"

namespace moe {

// Device error word written by bounded waits in the kernels (0 = none).
__device__ int g_device_error = 0;

namespace {
constexpr int kErrSelfTestTimeout = 0x1ff;

// One thread waits on a fresh mbarrier that nothing ever arrives at, with a clock budget of
// `budget` cycles; when the budget runs out it records kErrSelfTestTimeout and returns.
__global__ void selftest_wait_kernel(long long budget) {
    __shared__ uint64_t bar;
    __shared__ int never;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        never = 0;
        sm100::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !sm100::mbar_wait(&bar, 0, &never, budget))
        atomicCAS(&g_device_error, 0, kErrSelfTestTimeout);
}
}  // namespace

bool config_ok(const moe_config* c) {
    if (!c) return false;
    if (c->hidden <= 0 || c->inter <= 0 || c->n_experts <= 0 || c->n_group <= 0 ||
        c->topk_group <= 0 || c->top_k <= 0)
        return false;
    if (c->n_experts % c->n_group != 0 || c->n_experts / c->n_group < 2) return false;
    if (c->n_group > 32 || c->topk_group > c->n_group) return false;
    if (c->top_k > c->topk_group * (c->n_experts / c->n_group)) return false;
    if (c->n_experts > 1024 || c->top_k > 32) return false;
    if (c->has_shared != 0 && c->has_shared != 1) return false;
    if (c->mode != MOE_FP32 && c->mode != MOE_FP8_BLOCK && c->mode != MOE_MXFP8) return false;
    if (c->hidden % 128 != 0 || c->inter % 128 != 0) return false;
    return true;
}

static size_t align_up(size_t v) { return (v + 1023) & ~static_cast<size_t>(1023); }

WsLayout ws_layout(const moe_config& c, int64_t T) {
    WsLayout L{};
    const int64_t H = c.hidden, I = c.inter, E = c.n_experts, K = c.top_k, S = c.has_shared;
    const bool fp8 = (c.mode != MOE_FP32);
    const int64_t R = T * K + T * S;
    L.R = R;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
    L.xq = take(fp8 ? T * H : 0);
    L.xs = take(fp8 ? T * (H / 128) * 4 : 0);
    L.offs = take((E + 2) * 4);
    L.perm_tok = take(R * 4);
    L.row_of = take(T * K * 4);
    L.aq = take(fp8 ? R * H : R * H * 4);
    L.as = take(fp8 ? R * (H / 128) * 4 : 0);
    L.hq = take(fp8 ? R * I : R * I * 4);
    L.hs = take(fp8 ? R * (I / 128) * 4 : 0);
    L.yexp = take(fp8 ? R * H * 2 : R * H * 4);
    L.perm_scratch = take(permute_scratch_bytes(T, static_cast<int>(E)));
    L.gemm_scratch = take(fp8 ? tc_scratch_bytes(static_cast<int32_t>(E + S))
                              : gemm_scratch_bytes(static_cast<int32_t>(E + S), R, static_cast<int32_t>(2 * I),
                                                   MOE_EPI_SWIGLU_QUANT));
    L.total = o;
    return L;
}

}  // namespace moe

using namespace moe;

extern "C" const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: configuration not supported";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA launch or runtime error";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait expired";
    }
    return "unknown moe_status";
}

extern "C" moe_status moe_config_validate(const moe_config* cfg) {
    return config_ok(cfg) ? MOE_OK : MOE_ERR_INVALID_ARG;
}

extern "C" moe_status moe_workspace_size(const moe_config* cfg, int64_t T, size_t* bytes) {
    if (!config_ok(cfg) || T < 0 || !bytes) return MOE_ERR_INVALID_ARG;
    *bytes = ws_layout(*cfg, T).total;
    return MOE_OK;
}

extern "C" moe_status moe_device_error(int32_t* code) {
    if (!code) return MOE_ERR_INVALID_ARG;
    int v = 0;
    MOE_CUDA_CHECK(cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)));
    const int zero = 0;
    MOE_CUDA_CHECK(cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)));
    int32_t tc = 0, mx = 0, gate = 0, perm = 0, comb = 0;
    MOE_TRY(tc_read_and_clear_error(&tc));
    MOE_TRY(mx_read_and_clear_error(&mx));
    MOE_TRY(gate_read_and_clear_error(&gate));
    MOE_TRY(permute_read_and_clear_check(&perm));
    MOE_TRY(combine_read_and_clear_check(&comb));
    *code = v ? v : (tc ? tc : (mx ? mx : (gate ? gate : (perm ? perm : comb))));
    return MOE_OK;
}

extern "C" moe_status moe_selftest_wait_timeout(int64_t budget_cycles, moe_stream_t stream) {
    if (budget_cycles < 1 || budget_cycles > 4000000000LL) return MOE_ERR_INVALID_ARG;
    selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(budget_cycles);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

extern "C" moe_status moe_gate(const moe_config* cfg, int64_t T, const void* x, const void* Wg,
                               const float* bias, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, moe_stream_t stream) {
    if (!config_ok(cfg) || T < 0 || !counts) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !Wg || !bias || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
    return launch_gate(*cfg, T, x, Wg, bias, topk_idx, topk_w, counts, nullptr,
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" moe_status moe_gate_quant(const moe_config* cfg, int64_t T, const void* x, const void* Wg,
                                     const float* bias, int32_t* topk_idx, float* topk_w,
                                     int32_t* counts, uint8_t* xq, float* xs, moe_stream_t stream) {
    if (!config_ok(cfg) || T < 0 || !counts) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !Wg || !bias || !topk_idx || !topk_w || !xq || !xs)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (T > INT64_MAX / cfg->hidden)) return MOE_ERR_INVALID_ARG;
    return launch_gate_quant(*cfg, T, x, Wg, bias, topk_idx, topk_w, counts, xq, xs,
                             reinterpret_cast<cudaStream_t>(stream));
}

extern "C" moe_status moe_grouped_gemm_fp8(int32_t n_groups, const int32_t* offs, int64_t rows,
                                           int32_t N, int32_t Kdim, const uint8_t* A,
                                           const float* As, const uint8_t* W, const float* Ws,
                                           int32_t epilogue, void* out, float* out_s, void* ws,
                                           size_t ws_bytes, moe_stream_t stream) {
    if (n_groups < 1 || rows < 0 || N <= 0 || Kdim <= 0 || N % 128 || Kdim % 128)
        return MOE_ERR_INVALID_ARG;
    if (n_groups > kMaxGemmGroups) return MOE_ERR_UNSUPPORTED;  // the tile schedule lives in shared memory
    if (epilogue == MOE_EPI_SWIGLU_QUANT) {
        if (N % 256 != 0 || !out_s || !aligned16(out_s)) return MOE_ERR_INVALID_ARG;
    } else if (epilogue != MOE_EPI_STORE) {
        return MOE_ERR_INVALID_ARG;
    }
    if (!offs || !A || !As || !W || !Ws || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(As) || !aligned16(W) || !aligned16(Ws) || !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    (void)ws_bytes;  // the kernel builds its tile schedule in shared memory: no workspace
    if (rows == 0) return MOE_OK;
    return launch_grouped_gemm_fp8_tc(n_groups, offs, rows, N, Kdim, A, As, W, Ws, epilogue, out,
                                      out_s, ws, reinterpret_cast<cudaStream_t>(stream));
}

// Shared argument checks of the gathered grouped GEMMs.
static moe_status check_gather_args(int32_t n_groups, const int32_t* offs, int64_t rows, int32_t N, int32_t Kdim,
                                    const int32_t* perm_tok, int64_t T, const uint8_t* X, const float* Xs,
                                    const uint8_t* W, const float* Ws, int32_t epilogue, void* out, float* out_s) {
    if (n_groups < 1 || rows < 0 || T < 0 || N <= 0 || Kdim <= 0 || N % 128 || Kdim % 128) return MOE_ERR_INVALID_ARG;
    if (n_groups > kMaxGemmGroups) return MOE_ERR_UNSUPPORTED;
    if (epilogue == MOE_EPI_SWIGLU_QUANT) {
        if (N % 256 != 0 || !out_s || !aligned16(out_s)) return MOE_ERR_INVALID_ARG;
    } else if (epilogue != MOE_EPI_STORE) {
        return MOE_ERR_INVALID_ARG;
    }
    if (!offs || !perm_tok || !X || !Xs || !W || !Ws || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Xs) || !aligned16(W) || !aligned16(Ws) || !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

extern "C" moe_status moe_grouped_gemm_fp8_gather(int32_t n_groups, const int32_t* offs, int64_t rows, int32_t N,
                                                  int32_t Kdim, const int32_t* perm_tok, int64_t T,
                                                  const uint8_t* X, const float* Xs, const uint8_t* W,
                                                  const float* Ws, int32_t epilogue, void* out, float* out_s,
                                                  moe_stream_t stream) {
    MOE_TRY(check_gather_args(n_groups, offs, rows, N, Kdim, perm_tok, T, X, Xs, W, Ws, epilogue, out, out_s));
    if (rows == 0 || T == 0) return MOE_OK;
    return launch_grouped_gemm_fp8_tc(n_groups, offs, rows, N, Kdim, X, Xs, W, Ws, epilogue, out, out_s, nullptr,
                                      reinterpret_cast<cudaStream_t>(stream), perm_tok, T);
}

extern "C" moe_status moe_grouped_gemm_mxfp8_gather(int32_t n_groups, const int32_t* offs, int64_t rows, int32_t N,
                                                    int32_t Kdim, const int32_t* perm_tok, int64_t T,
                                                    const uint8_t* X, const float* Xs, const uint8_t* W,
                                                    const float* Ws, int32_t epilogue, void* out, float* out_s,
                                                    moe_stream_t stream) {
    MOE_TRY(check_gather_args(n_groups, offs, rows, N, Kdim, perm_tok, T, X, Xs, W, Ws, epilogue, out, out_s));
    if (rows == 0 || T == 0) return MOE_OK;
    return launch_grouped_gemm_mxf8(n_groups, offs, rows, N, Kdim, X, Xs, W, Ws, epilogue, out, out_s,
                                    reinterpret_cast<cudaStream_t>(stream), perm_tok, T);
}

extern "C" moe_status moe_forward(const moe_config* cfg, int64_t T, const void* x,
                                  const moe_weights* w, float* bias, int32_t update_bias,
                                  void* y, int32_t* topk_idx, float* topk_w, int32_t* counts,
                                  void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!config_ok(cfg) || T < 0 || !w || !counts || !ws || !bias) return MOE_ERR_INVALID_ARG;
    const moe_config& c = *cfg;
    const bool fp8 = (c.mode != MOE_FP32);
    const bool mx = (c.mode == MOE_MXFP8);
    if (!w->Wg || !w->W13 || !w->W2 || (fp8 && (!w->W13_s || !w->W2_s))) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !y || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ws) || (T > 0 && (!aligned16(x) || !aligned16(y)))) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c, T);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    char* base = static_cast<char*>(ws);
    const int64_t H = c.hidden, I = c.inter;
    const int32_t G = c.n_experts + c.has_shared;
    int32_t* offs = reinterpret_cast<int32_t*>(base + L.offs);
    int32_t* perm_tok = reinterpret_cast<int32_t*>(base + L.perm_tok);
    int32_t* row_of = reinterpret_cast<int32_t*>(base + L.row_of);
    void* gscratch = base + L.gemm_scratch;
    const size_t gbytes = L.total - L.gemm_scratch;

    // FP8 modes: from MOE_GATE_QUANT_MIN_TOKENS tokens up the gate also writes the 1x128
    // quantisation of x when its tensor-core kernel takes the shape (x is then read once);
    // otherwise the quantiser runs on its own below
    uint8_t* xq = fp8 ? reinterpret_cast<uint8_t*>(base + L.xq) : nullptr;
    float* xs = fp8 ? reinterpret_cast<float*>(base + L.xs) : nullptr;
    const bool fused = fp8 && T >= MOE_GATE_QUANT_MIN_TOKENS && gate_quant_supported(c) && aligned16(w->Wg);
    if (fused) MOE_TRY(moe_gate_quant(cfg, T, x, w->Wg, bias, topk_idx, topk_w, counts, xq, xs, stream));
    else MOE_TRY(moe_gate(cfg, T, x, w->Wg, bias, topk_idx, topk_w, counts, stream));
    if (update_bias) MOE_TRY(moe_bias_update(cfg, T, counts, bias, stream));
    if (T == 0) return MOE_OK;
    if (fp8) {
        uint8_t* aq = reinterpret_cast<uint8_t*>(base + L.aq);
        float* as = reinterpret_cast<float*>(base + L.as);
        uint8_t* hq = reinterpret_cast<uint8_t*>(base + L.hq);
        float* hs = reinterpret_cast<float*>(base + L.hs);
        void* yexp = base + L.yexp;
        if (!fused && mx) MOE_TRY(moe_quant_1x128_pow2(T, H, static_cast<const uint16_t*>(x), xq, xs, stream));
        else if (!fused) MOE_TRY(moe_quant_1x128(T, H, static_cast<const uint16_t*>(x), xq, xs, stream));
        // the permuted copy of the quantised rows: the grouped GEMM reads its A tiles with one TMA
        // box per K block (reading them straight from xq with tile::gather4, as
        // moe_grouped_gemm_fp8_gather does, measured twice as slow for the gate/up GEMM)
        MOE_TRY(moe_permute(cfg, T, topk_idx, counts, xq, xs, offs, perm_tok, row_of, aq, as, ws,
                            ws_bytes, stream));
        const int32_t N1 = static_cast<int32_t>(2 * I), N2 = static_cast<int32_t>(H);
        const uint8_t* W13 = static_cast<const uint8_t*>(w->W13);
        const uint8_t* W2 = static_cast<const uint8_t*>(w->W2);
        if (mx) {
            MOE_TRY(moe_grouped_gemm_mxfp8(G, offs, L.R, N1, N2, aq, as, W13, w->W13_s, MOE_EPI_SWIGLU_QUANT,
                                           hq, hs, stream));
            MOE_TRY(moe_grouped_gemm_mxfp8(G, offs, L.R, N2, static_cast<int32_t>(I), hq, hs, W2, w->W2_s,
                                           MOE_EPI_STORE, yexp, nullptr, stream));
        } else {
            MOE_TRY(moe_grouped_gemm_fp8(G, offs, L.R, N1, N2, aq, as, W13, w->W13_s, MOE_EPI_SWIGLU_QUANT,
                                         hq, hs, gscratch, gbytes, stream));
            MOE_TRY(moe_grouped_gemm_fp8(G, offs, L.R, N2, static_cast<int32_t>(I), hq, hs, W2, w->W2_s,
                                         MOE_EPI_STORE, yexp, nullptr, gscratch, gbytes, stream));
        }
        const void* yshared = c.has_shared ? static_cast<const char*>(yexp) + T * c.top_k * H * 2 : nullptr;
        MOE_TRY(moe_combine(cfg, T, yexp, row_of, topk_w, yshared, y, stream));
    } else {
        float* aq = reinterpret_cast<float*>(base + L.aq);
        float* h = reinterpret_cast<float*>(base + L.hq);
        float* yexp = reinterpret_cast<float*>(base + L.yexp);
        MOE_TRY(moe_permute(cfg, T, topk_idx, counts, x, nullptr, offs, perm_tok, row_of, aq,
                            nullptr, ws, ws_bytes, stream));
        MOE_TRY(moe_grouped_gemm_f32(G, offs, L.R, static_cast<int32_t>(2 * I), static_cast<int32_t>(H),
                                     aq, static_cast<const float*>(w->W13), MOE_EPI_SWIGLU_QUANT,
                                     h, gscratch, gbytes, stream));
        MOE_TRY(moe_grouped_gemm_f32(G, offs, L.R, static_cast<int32_t>(H), static_cast<int32_t>(I),
                                     h, static_cast<const float*>(w->W2), MOE_EPI_STORE, yexp,
                                     gscratch, gbytes, stream));
        const float* yshared = c.has_shared ? yexp + T * c.top_k * H : nullptr;
        MOE_TRY(moe_combine(cfg, T, yexp, row_of, topk_w, yshared, y, stream));
    }
    return MOE_OK;
}
