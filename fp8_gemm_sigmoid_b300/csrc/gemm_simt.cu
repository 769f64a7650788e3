// gemm_simt.cu -- grouped expert GEMM on the CUDA cores (FP32 FMA), used for the all-FP32
// layer, plus the tile scheduler prefix and the SwiGLU epilogue kernels shared by the
// grouped GEMMs.
//
// DeepSeek-V3 co-design teardown (wsisp.com) §5.1: FP8 operands with per-block scales applied
// during accumulation, FP32 accumulation.  Insights into DeepSeek-V3 précis §3.2: 1x128
// activation tiles and 128x128 weight blocks.  For group g (rows [offs[g], offs[g+1])):
//   out[r, n] = sum_kb (as[r,kb] * Ws[g, n/128, kb]) * sum_{k in kb} A[r,k] * W[g,n,k].
#include "common.cuh"
#include "internal.h"
#include "gemm.h"

namespace moe {

// tile_start[g] = number of kBM-row tiles of groups before g; tile_start[n_groups] = total.
__global__ void tile_prefix_kernel(int n_groups, int bm, const int32_t* __restrict__ offs,
                                   int32_t* __restrict__ tile_start) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int32_t run = 0;
    for (int g = 0; g < n_groups; ++g) {
        tile_start[g] = run;
        const int32_t cnt = offs[g + 1] - offs[g];
        run += (cnt + bm - 1) / bm;
    }
    tile_start[n_groups] = run;
}

namespace {

constexpr int kBM = 64, kBN = 64, kBK = 32, kThreads = 256;

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// A: [rows, Kd] FP32; W: [n_groups, N, Kd] FP32.  out: [rows, N] FP32.
__global__ void __launch_bounds__(kThreads)
grouped_gemm_f32_kernel(int n_groups, const int32_t* __restrict__ offs,
                        const int32_t* __restrict__ tile_start, int N, int Kd,
                        const float* __restrict__ A, const float* __restrict__ W,
                        float* __restrict__ out) {
    __shared__ float As[kBK][kBM + 4];
    __shared__ float Ws[kBK][kBN + 4];
    const int tile = blockIdx.x;
    if (tile >= tile_start[n_groups]) return;
    const int g = find_group(tile_start, n_groups, tile);
    const int64_t r0 = offs[g] + static_cast<int64_t>(tile - tile_start[g]) * kBM;
    const int64_t r_end = offs[g + 1];
    const int n0 = blockIdx.y * kBN;
    const float* Wg = W + static_cast<int64_t>(g) * N * Kd;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < Kd; k0 += kBK) {
        for (int i = tid; i < kBM * kBK; i += kThreads) {
            const int m = i / kBK, kk = i % kBK;
            const int64_t r = r0 + m;
            As[kk][m] = (r < r_end) ? A[r * Kd + k0 + kk] : 0.f;
            Ws[kk][m] = Wg[static_cast<int64_t>(n0 + m) * Kd + k0 + kk];
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kBK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Ws[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t r = r0 + ty * 4 + i;
        if (r < r_end)
            *reinterpret_cast<float4*>(out + r * N + n0 + tx * 4) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
}

// FP8 operands on the CUDA cores: the E4M3 codes are decoded to FP32 in shared memory; each
// 128-wide K block is accumulated separately and promoted with (as[r,kb] * Ws[g,nb,kb]).
// A: [rows, Kd] codes, As: [rows, Kd/128]; W: [n_groups, N, Kd], Ws: [n_groups, N/128, Kd/128].
// out: FP32 [rows, N] (to_bf16 = false) or BF16 [rows, N] (to_bf16 = true).
__global__ void __launch_bounds__(kThreads)
grouped_gemm_fp8_simt_kernel(int n_groups, const int32_t* __restrict__ offs,
                             const int32_t* __restrict__ tile_start, int N, int Kd,
                             const uint8_t* __restrict__ A, const float* __restrict__ As_,
                             const uint8_t* __restrict__ W, const float* __restrict__ Ws_,
                             void* __restrict__ out, bool to_bf16) {
    __shared__ float As[kBK][kBM + 4];
    __shared__ float Ws[kBK][kBN + 4];
    const int tile = blockIdx.x;
    if (tile >= tile_start[n_groups]) return;
    const int g = find_group(tile_start, n_groups, tile);
    const int64_t r0 = offs[g] + static_cast<int64_t>(tile - tile_start[g]) * kBM;
    const int64_t r_end = offs[g + 1];
    const int n0 = blockIdx.y * kBN;
    const int kblocks = Kd / 128;
    const uint8_t* Wg = W + static_cast<int64_t>(g) * N * Kd;
    const float* Wsg = Ws_ + (static_cast<int64_t>(g) * (N / 128) + n0 / 128) * kblocks;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float acc[4][4] = {};
    for (int kb = 0; kb < kblocks; ++kb) {
        float p[4][4] = {};
        for (int k0 = kb * 128; k0 < kb * 128 + 128; k0 += kBK) {
            // 64 rows x 32 codes per operand: thread tid loads 16 codes of A (tid < 128) or W
            const int op = tid / 128, t2 = tid % 128, m = t2 / 2, c16 = (t2 % 2) * 16;
            uint4 v;
            if (op == 0) {
                const int64_t r = r0 + m;
                v = (r < r_end) ? *reinterpret_cast<const uint4*>(A + r * Kd + k0 + c16)
                                : make_uint4(0u, 0u, 0u, 0u);
            } else {
                v = *reinterpret_cast<const uint4*>(Wg + static_cast<int64_t>(n0 + m) * Kd + k0 + c16);
            }
            float (*dst)[kBM + 4] = (op == 0) ? As : Ws;
            const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4)
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[c16 + w4 * 4 + i][m] = e4m3_to_f32((vw[w4] >> (8 * i)) & 0xffu);
            __syncthreads();
#pragma unroll 8
            for (int kk = 0; kk < kBK; ++kk) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Ws[kk][tx * 4 + i]; }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) p[i][j] = fmaf(a[i], b[j], p[i][j]);
            }
            __syncthreads();
        }
        const float sb = Wsg[kb];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t r = r0 + ty * 4 + i;
            const float sa = (r < r_end) ? As_[r * kblocks + kb] : 0.f;
            const float sc = sa * sb;
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(p[i][j], sc, acc[i][j]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t r = r0 + ty * 4 + i;
        if (r >= r_end) continue;
        if (to_bf16) {
            uint16_t* o = static_cast<uint16_t*>(out) + r * N + n0 + tx * 4;
            uint2 pk = make_uint2(f32_to_bf16_bits(acc[i][0]) | (uint32_t(f32_to_bf16_bits(acc[i][1])) << 16),
                                  f32_to_bf16_bits(acc[i][2]) | (uint32_t(f32_to_bf16_bits(acc[i][3])) << 16));
            *reinterpret_cast<uint2*>(o) = pk;
        } else {
            *reinterpret_cast<float4*>(static_cast<float*>(out) + r * N + n0 + tx * 4) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
    }
}

// h[r, j] = silu(gu[r, j]) * gu[r, I + j] for rows below offs[n_groups]; FP32 out.
__global__ void swiglu_f32_kernel(int64_t rows, int I, const int32_t* __restrict__ offs_end,
                                  const float* __restrict__ gu, float* __restrict__ h) {
    const int64_t R = *offs_end;
    const int64_t total = R * I;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / I;
        const int j = static_cast<int>(i % I);
        const float g = gu[r * 2 * I + j], u = gu[r * 2 * I + I + j];
        h[r * I + j] = silu_f32(g) * u;
    }
    (void)rows;
}

}  // namespace

// h = silu(g) * u in FP32, then 1x128 quantisation of h: 16 threads per tile, 8 values
// each; warp-uniform grid-stride loop over pairs of tiles.
__global__ void __launch_bounds__(256)
swiglu_quant_kernel(int I, const int32_t* __restrict__ offs_end, const float* __restrict__ gu,
                    uint8_t* __restrict__ hq, float* __restrict__ hs) {
    const int64_t R = *offs_end;
    const int tpr = I / 128;
    const int64_t n_tiles = R * tpr;
    const int sub = threadIdx.x & 15, half = (threadIdx.x >> 4) & 1;
    const int64_t n_pairs = (n_tiles + 1) / 2;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    for (int64_t pair = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
         pair < n_pairs; pair += nwarps) {
        const int64_t tile = pair * 2 + half;
        const bool valid = tile < n_tiles;
        const int64_t r = valid ? tile / tpr : 0;
        const int j0 = valid ? static_cast<int>(tile % tpr) * 128 + sub * 8 : 0;
        float h[8];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float g = valid ? gu[r * 2 * I + j0 + i] : 0.f;
            const float u = valid ? gu[r * 2 * I + I + j0 + i] : 0.f;
            h[i] = silu_f32(g) * u;
            amax = fmaxf(amax, fabsf(h[i]));
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        uint32_t p[4] = {0u, 0u, 0u, 0u};
        float scale = 1.f;
        if (amax != 0.f) {
            const float mul = __fdiv_rn(448.f, amax);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                p[i] = f32x2_to_e4m3x2(__fmul_rn(h[2 * i], mul), __fmul_rn(h[2 * i + 1], mul));
            scale = __fdiv_rn(amax, 448.f);
        }
        if (valid) {
            *reinterpret_cast<uint2*>(hq + r * I + j0) = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
            if (sub == 0) hs[r * tpr + j0 / 128] = scale;
        }
    }
}

moe_status launch_grouped_gemm_fp8_simt(int32_t n_groups, const int32_t* offs, int64_t rows,
                                        int32_t N, int32_t Kd, const uint8_t* A, const float* As,
                                        const uint8_t* W, const float* Ws, int32_t epilogue,
                                        void* out, float* out_s, void* ws, cudaStream_t s) {
    int32_t* tile_start = static_cast<int32_t*>(ws);
    float* gu = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                         (static_cast<size_t>(n_groups) + 1 + 255) / 256 * 1024);
    MOE_TRY(launch_tile_prefix(n_groups, kBM, offs, tile_start, s));
    const int64_t max_tiles = ceil_div(rows, kBM) + n_groups;
    dim3 grid(static_cast<unsigned>(max_tiles), static_cast<unsigned>(N / kBN));
    const bool store = (epilogue == MOE_EPI_STORE);
    grouped_gemm_fp8_simt_kernel<<<grid, kThreads, 0, s>>>(n_groups, offs, tile_start, N, Kd, A, As,
                                                          W, Ws, store ? out : gu, store);
    MOE_LAUNCH_CHECK();
    if (!store) {
        swiglu_quant_kernel<<<148 * 8, 256, 0, s>>>(N / 2, offs + n_groups, gu,
                                                    static_cast<uint8_t*>(out), out_s);
        MOE_LAUNCH_CHECK();
    }
    return MOE_OK;
}

moe_status launch_tile_prefix(int n_groups, int bm, const int32_t* offs, int32_t* tile_start,
                              cudaStream_t s) {
    tile_prefix_kernel<<<1, 32, 0, s>>>(n_groups, bm, offs, tile_start);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

// Scratch of one grouped-GEMM call: the tile prefix and, for the SwiGLU epilogue, the FP32
// gate/up outputs [rows, N].
size_t gemm_scratch_bytes(int32_t n_groups, int64_t rows, int32_t N, int32_t epilogue) {
    const size_t prefix = (static_cast<size_t>(n_groups) + 1 + 255) / 256 * 1024;
    if (epilogue != MOE_EPI_SWIGLU_QUANT) return prefix;
    return prefix + static_cast<size_t>(rows) * N * sizeof(float);
}

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_grouped_gemm_f32(int32_t n_groups, const int32_t* offs, int64_t rows,
                                           int32_t N, int32_t Kdim, const float* A, const float* W,
                                           int32_t epilogue, float* out, void* ws,
                                           size_t ws_bytes, moe_stream_t stream) {
    if (n_groups < 1 || rows < 0 || N <= 0 || Kdim <= 0 || N % 128 || Kdim % 128) return MOE_ERR_INVALID_ARG;
    if (epilogue != MOE_EPI_SWIGLU_QUANT && epilogue != MOE_EPI_STORE) return MOE_ERR_INVALID_ARG;
    if (!offs || !A || !W || !out || !ws || !aligned16(A) || !aligned16(W) || !aligned16(out) || !aligned16(ws))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < gemm_scratch_bytes(n_groups, rows, N, epilogue)) return MOE_ERR_WORKSPACE;
    if (rows == 0) return MOE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t* tile_start = static_cast<int32_t*>(ws);
    float* gu = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                         (static_cast<size_t>(n_groups) + 1 + 255) / 256 * 1024);
    MOE_TRY(launch_tile_prefix(n_groups, kBM, offs, tile_start, s));
    const int64_t max_tiles = ceil_div(rows, kBM) + n_groups;
    dim3 grid(static_cast<unsigned>(max_tiles), static_cast<unsigned>(N / kBN));
    float* dst = (epilogue == MOE_EPI_STORE) ? out : gu;
    grouped_gemm_f32_kernel<<<grid, kThreads, 0, s>>>(n_groups, offs, tile_start, N, Kdim, A, W, dst);
    MOE_LAUNCH_CHECK();
    if (epilogue == MOE_EPI_SWIGLU_QUANT) {
        swiglu_f32_kernel<<<148 * 8, 256, 0, s>>>(rows, N / 2, offs + n_groups, gu, out);
        MOE_LAUNCH_CHECK();
    }
    return MOE_OK;
}
