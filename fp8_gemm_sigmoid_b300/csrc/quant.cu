// quant.cu -- a2: fine-grained FP8 quantisation (Insights into DeepSeek-V3 précis, §3.2:
// activations in 1x128 tiles, weights in 128x128 blocks, one FP32 scale each).
//
// Rule (both granularities): amax = max |v| over the tile; scale = amax / 448;
// code = E4M3(v * (448 / amax)) rounded to nearest even and saturated to +-448;
// amax == 0 gives scale 1 and all-zero codes.  Divisions and the product are IEEE FP32.
// Power-of-two mode (the scales the précis asks tensor cores to take natively, §3.2; the
// block-scaled MMA reads them as 8-bit exponents): scale = 2^e with e the smallest integer
// such that 448 * 2^e >= amax, clamped to [-127, 127], and code = E4M3(v * 2^-e), an exact
// scaling, so no value saturates.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// 16 threads per 1x128 tile, 8 BF16 (16 bytes) per thread; each warp takes two tiles per
// step of a grid-stride loop whose trip count is uniform across the warp.
template <bool kPow2>
__global__ void __launch_bounds__(256)
quant_1x128_kernel(int64_t n_tiles, const uint4* __restrict__ x, uint2* __restrict__ q,
                   float* __restrict__ s) {
    const int sub = threadIdx.x & 15;
    const int half = (threadIdx.x >> 4) & 1;
    const int64_t n_pairs = (n_tiles + 1) / 2;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
    for (int64_t pair = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
         pair < n_pairs; pair += nwarps) {
        const int64_t tile = pair * 2 + half;  // tile = row * (cols/128) + block
        const bool valid = tile < n_tiles;
        uint4 v = valid ? x[tile * 16 + sub] : make_uint4(0u, 0u, 0u, 0u);
        float f[8];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        uint2 out;
        float scale;
        if (amax == 0.f) {
            out = make_uint2(0u, 0u);
            scale = 1.f;
        } else if (kPow2) {
            const int e = pow2_exponent(amax);
            uint32_t p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                p[i] = f32x2_to_e4m3x2(scale_pow2(f[2 * i], e), scale_pow2(f[2 * i + 1], e));
            out = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
            scale = exp2_int(e);
        } else {
            const float mul = __fdiv_rn(448.f, amax);
            uint32_t p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                p[i] = f32x2_to_e4m3x2(__fmul_rn(f[2 * i], mul), __fmul_rn(f[2 * i + 1], mul));
            out = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
            scale = __fdiv_rn(amax, 448.f);
        }
        if (valid) {
            q[tile * 16 + sub] = out;
            if (sub == 0) s[tile] = scale;
        }
    }
}

// One CTA per 128x128 block: amax over the block, then encode.  w is [n, rows, cols].
template <bool kPow2>
__global__ void __launch_bounds__(256)
quant_128x128_kernel(int64_t rows, int64_t cols, const uint16_t* __restrict__ w,
                     uint8_t* __restrict__ q, float* __restrict__ s) {
    __shared__ float red[8];
    const int64_t rb = rows / 128, cb = cols / 128;
    const int64_t blk = blockIdx.x;  // m * rb * cb + i * cb + j
    const int64_t m = blk / (rb * cb), i = (blk / cb) % rb, j = blk % cb;
    const int64_t base = m * rows * cols + i * 128 * cols + j * 128;
    const int tid = threadIdx.x;
    const int c16 = tid & 15;       // 16-byte chunk within the 256-byte row
    const int r0 = tid >> 4;        // 16 rows per pass
    float amax = 0.f;
    for (int r = r0; r < 128; r += 16) {
        uint4 v = *reinterpret_cast<const uint4*>(w + base + r * cols + c16 * 8);
        const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            amax = fmaxf(amax, fabsf(__uint_as_float(ww[k] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(ww[k] & 0xffff0000u)));
        }
    }
    amax = warp_max(amax);
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int k = 1; k < 8; ++k) amax = fmaxf(amax, red[k]);
    const bool zero = (amax == 0.f);
    const float mul = (zero || kPow2) ? 0.f : __fdiv_rn(448.f, amax);
    const int e = (zero || !kPow2) ? 0 : pow2_exponent(amax);
    for (int r = r0; r < 128; r += 16) {
        uint4 v = *reinterpret_cast<const uint4*>(w + base + r * cols + c16 * 8);
        const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
        uint32_t p[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float lo = __uint_as_float(ww[k] << 16), hi = __uint_as_float(ww[k] & 0xffff0000u);
            if (zero) p[k] = 0u;
            else if (kPow2) p[k] = f32x2_to_e4m3x2(scale_pow2(lo, e), scale_pow2(hi, e));
            else p[k] = f32x2_to_e4m3x2(__fmul_rn(lo, mul), __fmul_rn(hi, mul));
        }
        *reinterpret_cast<uint2*>(q + base + r * cols + c16 * 8) =
            make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
    }
    if (tid == 0) s[blk] = zero ? 1.f : (kPow2 ? exp2_int(e) : __fdiv_rn(amax, 448.f));
}

}  // namespace
}  // namespace moe

using namespace moe;

namespace {

moe_status quant_1x128(bool pow2, int64_t rows, int64_t cols, const uint16_t* x, uint8_t* q, float* s,
                       moe_stream_t stream) {
    if (rows < 0 || cols <= 0 || cols % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!x || !q || !s || !aligned16(x) || !aligned16(q) || !aligned16(s)) return MOE_ERR_INVALID_ARG;
    const int64_t tiles = rows * (cols / 128);
    const int64_t blocks = ceil_div(tiles, 16);  // 16 tiles per 256-thread CTA
    const unsigned grid = static_cast<unsigned>(blocks < 148 * 16 ? blocks : 148 * 16);
    auto k = pow2 ? quant_1x128_kernel<true> : quant_1x128_kernel<false>;
    k<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        tiles, reinterpret_cast<const uint4*>(x), reinterpret_cast<uint2*>(q), s);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

moe_status quant_128x128(bool pow2, int64_t n_mats, int64_t rows, int64_t cols, const uint16_t* w,
                         uint8_t* q, float* s, moe_stream_t stream) {
    if (n_mats < 0 || rows <= 0 || cols <= 0 || rows % 128 != 0 || cols % 128 != 0)
        return MOE_ERR_INVALID_ARG;
    if (n_mats == 0) return MOE_OK;
    if (!w || !q || !s || !aligned16(w) || !aligned16(q) || !aligned16(s)) return MOE_ERR_INVALID_ARG;
    const int64_t blocks = n_mats * (rows / 128) * (cols / 128);
    if (blocks > 0x7fffffffLL) return MOE_ERR_INVALID_ARG;
    auto k = pow2 ? quant_128x128_kernel<true> : quant_128x128_kernel<false>;
    k<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(rows, cols, w, q, s);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_quant_1x128(int64_t rows, int64_t cols, const uint16_t* x, uint8_t* q,
                                      float* s, moe_stream_t stream) {
    return quant_1x128(false, rows, cols, x, q, s, stream);
}

extern "C" moe_status moe_quant_1x128_pow2(int64_t rows, int64_t cols, const uint16_t* x, uint8_t* q,
                                           float* s, moe_stream_t stream) {
    return quant_1x128(true, rows, cols, x, q, s, stream);
}

extern "C" moe_status moe_quant_128x128(int64_t n_mats, int64_t rows, int64_t cols,
                                        const uint16_t* w, uint8_t* q, float* s,
                                        moe_stream_t stream) {
    return quant_128x128(false, n_mats, rows, cols, w, q, s, stream);
}

extern "C" moe_status moe_quant_128x128_pow2(int64_t n_mats, int64_t rows, int64_t cols,
                                             const uint16_t* w, uint8_t* q, float* s,
                                             moe_stream_t stream) {
    return quant_128x128(true, n_mats, rows, cols, w, q, s, stream);
}
