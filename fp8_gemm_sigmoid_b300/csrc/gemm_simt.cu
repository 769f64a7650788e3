// gemm_simt.cu -- the grouped expert GEMM of the all-FP32 layer on the CUDA cores (FP32 FMA,
// no quantisation) and its SwiGLU epilogue.  For group g (rows [offs[g], offs[g+1])):
//   out[r, n] = sum_k A[r, k] * W[g, n, k]   (FP32 accumulation).
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
