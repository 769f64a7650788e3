// combine.cu -- a7: weighted combine of the expert rows plus the shared expert, and a8: the
// load-driven selection-bias update.
//
// DeepSeek-V3 co-design teardown (wsisp.com) §2.3: after the experts run, each token's rows
// come back and are summed with its routing weights; Insights into DeepSeek-V3 précis §3.1:
// the combine payload is BF16.  Per token and column, in FP32 and slot order:
//   y = sum_k w[t,k] * yexp[row_of[t,k]] (+ yshared[t] for the shared expert),
// each term a separate FP32 multiply and add, rounded once to the output type.  A slot whose
// row lies outside [0, T*K) (row_of = -1: an expert id the permutation dropped) adds nothing.
#include "common.cuh"
#include "internal.h"

namespace moe {

// Check word of the MOE_CHECKS build (0 = none): 0x302, a combine row outside [-1, T*K)
// (-1 marks a dropped slot); 0x303, a gathered row index past the source rows.
__device__ int g_combine_check = 0;

moe_status combine_read_and_clear_check(int32_t* code) {
    MOE_CUDA_CHECK(read_and_clear_word(g_combine_check, code));
    return MOE_OK;
}

namespace {

// One thread per (token, 8 BF16 columns): 16-byte gathered loads, 16-byte store.
__global__ void __launch_bounds__(256)
combine_bf16_kernel(int64_t T, int H, int K, const uint16_t* __restrict__ yexp,
                    const int32_t* __restrict__ row_of, const float* __restrict__ w,
                    const uint16_t* __restrict__ yshared, uint16_t* __restrict__ y) {
    const int chunks = H / 8;
    const int64_t total = T * chunks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / chunks;
        const int ch = static_cast<int>(i % chunks);
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        for (int k = 0; k < K; ++k) {
            const int64_t r = row_of[t * K + k];
            if (r < 0 || r >= T * K) {  // dropped slot (-1); anything else is a caller's error
                (void)MOE_DCHECK(g_combine_check, r == -1, 0x302);
                continue;
            }
            const float wk = w[t * K + k];
            uint4 v = *reinterpret_cast<const uint4*>(yexp + r * H + ch * 8);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[2 * j] = __fadd_rn(acc[2 * j], __fmul_rn(wk, __uint_as_float(u[j] << 16)));
                acc[2 * j + 1] =
                    __fadd_rn(acc[2 * j + 1], __fmul_rn(wk, __uint_as_float(u[j] & 0xffff0000u)));
            }
        }
        if (yshared) {
            uint4 v = *reinterpret_cast<const uint4*>(yshared + t * H + ch * 8);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[2 * j] = __fadd_rn(acc[2 * j], __uint_as_float(u[j] << 16));
                acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], __uint_as_float(u[j] & 0xffff0000u));
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[j] = static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * j])) |
                   (static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * j + 1])) << 16);
        *reinterpret_cast<uint4*>(y + t * H + ch * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// The same for 4 <= K <= 8, with every load of a token's slots issued before any of them is
// used: the slots' row indices and weights first, then up to eight 16-byte row loads and the
// shared expert's, so that a thread keeps nine row loads in flight instead of one.  The sums run
// in slot order with the same operations, so the result is the general kernel's bit for bit.
// (For K = 1 or 2 the general kernel's higher occupancy wins: measured on the top-1 layer.)
__global__ void __launch_bounds__(256)
combine_bf16_k8_kernel(int64_t T, int H, int K, const uint16_t* __restrict__ yexp,
                       const int32_t* __restrict__ row_of, const float* __restrict__ w,
                       const uint16_t* __restrict__ yshared, uint16_t* __restrict__ y) {
    constexpr int kMaxK = 8;
    const int chunks = H / 8;
    const int64_t total = T * chunks;
    const int64_t rows = T * K;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / chunks;
        const int ch = static_cast<int>(i % chunks);
        int64_t r[kMaxK];
        float wk[kMaxK];
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            r[k] = k < K ? row_of[t * K + k] : -1;
            wk[k] = k < K ? w[t * K + k] : 0.f;
        }
        uint4 v[kMaxK];
        bool use[kMaxK];
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            use[k] = k < K && r[k] >= 0 && r[k] < rows;
            (void)MOE_DCHECK(g_combine_check, k >= K || use[k] || r[k] == -1, 0x302);
            v[k] = use[k] ? *reinterpret_cast<const uint4*>(yexp + r[k] * H + ch * 8) : make_uint4(0u, 0u, 0u, 0u);
        }
        const uint4 vs = yshared ? *reinterpret_cast<const uint4*>(yshared + t * H + ch * 8) : make_uint4(0u, 0u, 0u, 0u);
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            if (!use[k]) continue;  // a dropped slot adds nothing
            const uint32_t u[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[2 * j] = __fadd_rn(acc[2 * j], __fmul_rn(wk[k], __uint_as_float(u[j] << 16)));
                acc[2 * j + 1] =
                    __fadd_rn(acc[2 * j + 1], __fmul_rn(wk[k], __uint_as_float(u[j] & 0xffff0000u)));
            }
        }
        if (yshared) {
            const uint32_t u[4] = {vs.x, vs.y, vs.z, vs.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[2 * j] = __fadd_rn(acc[2 * j], __uint_as_float(u[j] << 16));
                acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], __uint_as_float(u[j] & 0xffff0000u));
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            o[j] = static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * j])) |
                   (static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * j + 1])) << 16);
        *reinterpret_cast<uint4*>(y + t * H + ch * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// FP32 rows: one thread per (token, 4 columns).
__global__ void __launch_bounds__(256)
combine_f32_kernel(int64_t T, int H, int K, const float* __restrict__ yexp,
                   const int32_t* __restrict__ row_of, const float* __restrict__ w,
                   const float* __restrict__ yshared, float* __restrict__ y) {
    const int chunks = H / 4;
    const int64_t total = T * chunks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / chunks;
        const int ch = static_cast<int>(i % chunks);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < K; ++k) {
            const int64_t r = row_of[t * K + k];
            if (r < 0 || r >= T * K) {  // dropped slot (-1); anything else is a caller's error
                (void)MOE_DCHECK(g_combine_check, r == -1, 0x302);
                continue;
            }
            const float wk = w[t * K + k];
            float4 v = *reinterpret_cast<const float4*>(yexp + r * H + ch * 4);
            acc.x = __fadd_rn(acc.x, __fmul_rn(wk, v.x));
            acc.y = __fadd_rn(acc.y, __fmul_rn(wk, v.y));
            acc.z = __fadd_rn(acc.z, __fmul_rn(wk, v.z));
            acc.w = __fadd_rn(acc.w, __fmul_rn(wk, v.w));
        }
        if (yshared) {
            float4 v = *reinterpret_cast<const float4*>(yshared + t * H + ch * 4);
            acc.x = __fadd_rn(acc.x, v.x);
            acc.y = __fadd_rn(acc.y, v.y);
            acc.z = __fadd_rn(acc.z, v.z);
            acc.w = __fadd_rn(acc.w, v.w);
        }
        *reinterpret_cast<float4*>(y + t * H + ch * 4) = acc;
    }
}

// b_i += 1e-3 * sign(T*K - E*counts[i]) (the sign of mean_load - load_i, in integers).
__global__ void bias_update_kernel(int E, int64_t T, int K, const int32_t* __restrict__ counts,
                                   float* __restrict__ bias) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int64_t d = T * K - static_cast<int64_t>(E) * counts[e];
        const int sgn = (d > 0) - (d < 0);
        bias[e] = __fadd_rn(bias[e], __fmul_rn(1e-3f, static_cast<float>(sgn)));
    }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_combine(const moe_config* cfg, int64_t T, const void* yexp,
                                  const int32_t* row_of, const float* topk_w,
                                  const void* yshared, void* y, moe_stream_t stream) {
    if (!config_ok(cfg) || T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!yexp || !row_of || !topk_w || !y || !aligned16(yexp) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    if (cfg->has_shared ? (!yshared || !aligned16(yshared)) : (yshared != nullptr))
        return MOE_ERR_INVALID_ARG;
    const moe_config& c = *cfg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t per = (c.mode == MOE_FP32) ? c.hidden / 4 : c.hidden / 8;
    const int64_t blocks = ceil_div(T * per, 256);
    const unsigned grid = static_cast<unsigned>(blocks < 148 * 16 ? blocks : 148 * 16);
    if (c.mode == MOE_FP32)
        combine_f32_kernel<<<grid, 256, 0, s>>>(T, c.hidden, c.top_k, static_cast<const float*>(yexp),
                                                row_of, topk_w, static_cast<const float*>(yshared),
                                                static_cast<float*>(y));
    else if (c.top_k >= 4 && c.top_k <= 8)
        combine_bf16_k8_kernel<<<grid, 256, 0, s>>>(T, c.hidden, c.top_k, static_cast<const uint16_t*>(yexp),
                                                    row_of, topk_w, static_cast<const uint16_t*>(yshared),
                                                    static_cast<uint16_t*>(y));
    else
        combine_bf16_kernel<<<grid, 256, 0, s>>>(T, c.hidden, c.top_k, static_cast<const uint16_t*>(yexp),
                                                 row_of, topk_w, static_cast<const uint16_t*>(yshared),
                                                 static_cast<uint16_t*>(y));
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

extern "C" moe_status moe_bias_update(const moe_config* cfg, int64_t T, const int32_t* counts,
                                      float* bias, moe_stream_t stream) {
    if (!config_ok(cfg) || T < 0 || !counts || !bias) return MOE_ERR_INVALID_ARG;
    bias_update_kernel<<<1, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        cfg->n_experts, T, cfg->top_k, counts, bias);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

// ---------------------------------------------------------------------------------------
// Row gather for the expert-parallel dispatch: dst[r] = src[idx[r]] (a zero row where
// idx[r] < 0), row_bytes a multiple of 16; one thread per 16-byte chunk.
// ---------------------------------------------------------------------------------------
namespace moe {
namespace {
__global__ void __launch_bounds__(256)
gather_rows_kernel(int64_t n_rows, int64_t chunks, const int32_t* __restrict__ idx,
                   const uint4* __restrict__ src, uint4* __restrict__ dst) {
    const int64_t total = n_rows * chunks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / chunks, c = i - r * chunks;
        const int32_t s = idx[r];
        dst[i] = s < 0 ? make_uint4(0u, 0u, 0u, 0u) : src[static_cast<int64_t>(s) * chunks + c];
    }
}
}  // namespace
}  // namespace moe

extern "C" moe_status moe_gather_rows(int64_t n_rows, int64_t row_bytes, const int32_t* idx, const void* src,
                                      void* dst, moe_stream_t stream) {
    if (n_rows < 0 || row_bytes <= 0 || row_bytes % 16) return MOE_ERR_INVALID_ARG;
    if (n_rows == 0) return MOE_OK;
    if (!idx || !src || !dst || !aligned16(src) || !aligned16(dst)) return MOE_ERR_INVALID_ARG;
    const int64_t chunks = row_bytes / 16;
    const int64_t blocks = ceil_div(n_rows * chunks, 256);
    const unsigned grid = static_cast<unsigned>(blocks < 148 * 16 ? blocks : 148 * 16);
    gather_rows_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        n_rows, chunks, idx, static_cast<const uint4*>(src), static_cast<uint4*>(dst));
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}
